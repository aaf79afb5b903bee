// Warmup mode on the 5th-generation tensor cores (d = d_I = 128, gs = 8).
//
// "MSA" study note 4-4 "Indexer warmup" (dense main branch, index branch
// trained against the full-context teacher), 4-2 (teacher = mean over the
// GQA group's heads of the main-branch probabilities) and 4-3 (teacher
// detached; the KL reaches only q^I and k^I).  Per row (t, g), over every key
// j <= t:
//   pbar_j = mean_h exp(scale q_h.k_j - lse_h),  zI_j = q^I.k^I_j / sqrt(d_I),
//   pI_j = exp(zI_j - lse^I),  KL = sum_j pbar_j (ln pbar_j - ln pI_j),
//   dzI_j = w (pI_j - pbar_j),
//   dq^I = sum_j dzI_j k^I_j / sqrt(d_I),  dk^I_j += dzI_j q^I / sqrt(d_I).
//
// Index gradient, key-outer: one CTA per (128-key tile, group), heaviest key
// tiles first, walking the query tiles of 16 positions x 8 heads that can see
// its keys.  Per query tile:
//   S^T = K Q^T    (M = keys, N = 128 rows = 16 positions x 8 heads, K = d)
//   Z^T = K^I Q^I^T (M = keys, N = 16 positions, K = d_I)
// into TMEM; each thread owns one key (TMEM lane), so a position's 8 head
// probabilities are 8 consecutive columns of its own row and the teacher is
// a sum of 8 registers, with no exchange between threads.  It forms dzI for
// the 16 positions, writes it (bf16) to TMEM (the A operand of dk^I) and to a
// K-major shared tile (the B operand of dq^I), and adds its KL terms;
//   dk^I  += dzI^T Q^I   (A from TMEM, Q^I as MN-major B), accumulated in
//                         TMEM over every query tile of the CTA and written
//                         once at the end;
//   dq^I^T = K^I^T dzI^T (K^I as MN-major A, M = d_I, N = 16 positions),
//                         added to dq^I with fp32 reductions (32 consecutive
//                         dims per warp instruction).
// The next query tile's rows arrive by cp.async while this one computes.  The
// main scores are computed once per (key, query) pair here; the forward pass
// keeps its own.
#include <math.h>

#include "msa_sm100.cuh"

namespace msa {

namespace {

using namespace sm100;

namespace wtc {
constexpr int kKeys = 128;   // keys of a CTA
constexpr int kPos = 16;     // positions of a query tile
constexpr int kRows = 128;   // 16 positions x 8 heads
constexpr int kThreads = 256;
constexpr int kChunk128 = 128 * 128;  // one 64-column chunk of a 128-row bf16 tile, bytes
constexpr int kTile128 = 2 * kChunk128;
constexpr int kChunk16 = 16 * 128;    // one 64-column chunk of a 16-row bf16 tile
constexpr int kTile16 = 2 * kChunk16;
constexpr int kK = 0, kKI = kTile128, kQ = 2 * kTile128;  // Q: two buffers
constexpr int kQI = 4 * kTile128;                           // Q^I: two buffers
constexpr int kDZ = kQI + 2 * kTile16;                      // dzI [16 positions][128 keys], K-major
constexpr int kBar = kDZ + kTile16;
constexpr int kBytes = 1024 + kBar + 64;
// TMEM columns: S^T, Z^T, dq^I^T, dzI^T (A operand, bf16 packed), dk^I
constexpr uint32_t kTS = 0, kTZ = 128, kTDQ = 160, kTDZ = 192, kTDK = 256;
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128);
constexpr uint32_t kIdescZ = idesc_bf16_f32(128, 16);
constexpr uint32_t kIdescDK = idesc_bf16_f32(128, 128) | (1u << 16);  // B MN-major
constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, 16) | (1u << 15);   // A MN-major
// Byte offset of element (row r, column c) of a 128B-swizzled K-major bf16
// tile whose 64-column chunks are `chunk` bytes apart (8-row groups 1 KB apart).
__device__ __forceinline__ uint32_t off(int r, int c, int chunk) {
  return (uint32_t)((c >> 6) * chunk + (r >> 3) * 1024 + (r & 7) * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) +
                    ((c & 7) << 1));
}
__device__ __forceinline__ void red_add(float* p, float a) {
  asm volatile("red.global.add.f32 [%0], %1;\n" ::"l"(p), "f"(a) : "memory");
}
__device__ __forceinline__ void red_add4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void reg_fence8(uint32_t (&r)[8]) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]));
}
__device__ __forceinline__ void tmem_st_x4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
}  // namespace wtc

__global__ void __launch_bounds__(wtc::kThreads, 1) warmup_grad_tc_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ kc, const uint16_t* __restrict__ q_idx,
    const uint16_t* __restrict__ k_idx, const float* __restrict__ lse, const float* __restrict__ lseI, int64_t N,
    int H_q, int G, float scale, float w_kl, float* __restrict__ dq_idx, float* __restrict__ dk_idx,
    float* __restrict__ kl, DeviceStatus* st) {
  using namespace wtc;
  constexpr int D = 128, DI = 128;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float lse2_s[kRows];   // main lse of each tile row, log2 units
  __shared__ float lseI2_s[kPos];   // lse^I of each position, log2 units
  __shared__ int32_t tpos_s[kPos];  // position of each tile position, -1 past N
  __shared__ float kl_s[8][8];      // per warp, the KL sums of its warpgroup's 8 positions
  const uint32_t bar_s = sb + kBar, bar_q = sb + kBar + 8, bar_drain = sb + kBar + 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;  // TMEM lane quadrant; positions 8 half .. 8 half + 7
  const int g = blockIdx.x;
  const int64_t j0 = (int64_t)blockIdx.y * kKeys;  // key tiles in launch order: the heaviest first
  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_q, 1);
    mbar_init(bar_drain, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;
  const float kLog2e = 1.4426950408889634f;
  const float sl2 = scale * kLog2e;             // main scores -> log2 units
  const float sI = 1.0f / sqrtf((float)DI);
  const float sI2 = sI * kLog2e;                // index logits -> log2 units
  const float kLn2 = 0.69314718055994530942f;

  // the CTA's keys: K (group g) and K^I, 128 x 128 each
  for (int i = tid; i < kKeys * 16; i += kThreads) {
    const int r = i >> 4, c = (i & 15) * 8;
    const int64_t j = j0 + r;
    const bool ok = j < N;
    cp_async_16(sm + kK + off(r, c, kChunk128), ok ? kc + (j * G + g) * D + c : kc, ok ? 16 : 0);
    cp_async_16(sm + kKI + off(r, c, kChunk128), ok ? k_idx + j * DI + c : k_idx, ok ? 16 : 0);
  }
  // rows of query tile qt into buffer b: Q rows r = 8 p + h (position p, head g*8 + h), Q^I rows p
  auto issue_q = [&](int64_t qt, int b) {
    const int64_t t0 = qt * kPos;
#pragma unroll
    for (int m = 0; m < kRows * 16 / kThreads; ++m) {
      const int i = tid + m * kThreads;
      const int r = i >> 4, c = (i & 15) * 8;
      const int64_t t = t0 + (r >> 3);
      const bool ok = t < N;
      cp_async_16(sm + kQ + b * kTile128 + off(r, c, kChunk128),
                  ok ? q + (t * H_q + (int64_t)g * 8 + (r & 7)) * D + c : q, ok ? 16 : 0);
    }
    {
      const int r = tid >> 4, c = (tid & 15) * 8;  // 16 rows x 16 units = 256 threads
      const int64_t t = t0 + r;
      const bool ok = t < N;
      cp_async_16(sm + kQI + b * kTile16 + off(r, c, kChunk16), ok ? q_idx + (t * G + g) * DI + c : q_idx,
                  ok ? 16 : 0);
    }
  };
  // row info of query tile qt into registers (stored to shared memory when the tile starts)
  float nt_lse = 0.f, nt_lseI = 0.f;
  int32_t nt_t = -1;
  auto load_row_info = [&](int64_t qt) {
    const int64_t t0 = qt * kPos;
    if (tid < kRows) {
      const int64_t t = t0 + (tid >> 3);
      nt_lse = t < N ? __ldg(lse + ((int64_t)g * 8 + (tid & 7)) * N + t) : 0.f;
    } else if (tid < kRows + kPos) {
      const int64_t t = t0 + (tid - kRows);
      nt_t = t < N ? (int32_t)t : -1;
      nt_lseI = t < N ? __ldg(lseI + (int64_t)g * N + t) : 0.f;
    }
  };
  const int64_t n_qt = (N + kPos - 1) / kPos;
  const int64_t qt0 = j0 / kPos;  // the first query tile with a position >= j0
  issue_q(qt0, 0);
  cp_async_commit();
  load_row_info(qt0);
  bool issued = false;
  uint32_t nt = 0;
  for (int64_t qt = qt0; qt < n_qt; ++qt, ++nt) {
    const int buf = (int)(nt & 1);
    if (tid < kRows) {
      lse2_s[tid] = nt_lse * kLog2e;
    } else if (tid < kRows + kPos) {
      tpos_s[tid - kRows] = nt_t;
      lseI2_s[tid - kRows] = nt_lseI * kLog2e;
    }
    cp_async_wait<0>();  // this tile's rows (and, at the first tile, the CTA's keys)
    fence_proxy_async_smem();
    __syncthreads();
    const uint32_t qb = sb + kQ + buf * kTile128, qib = sb + kQI + buf * kTile16;
    // ---- S^T and Z^T
    if (warp == 0 && lane == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int c = ks >> 2, kk = ks & 3;
        mma_bf16_ss(tmem + kTS, umma_desc_kmajor(sb + kK + c * kChunk128 + kk * 32, 128),
                    umma_desc_kmajor(qb + c * kChunk128 + kk * 32, 128), kIdescS, ks > 0);
        mma_bf16_ss(tmem + kTZ, umma_desc_kmajor(sb + kKI + c * kChunk128 + kk * 32, 128),
                    umma_desc_kmajor(qib + c * kChunk16 + kk * 32, 128), kIdescZ, ks > 0);
      }
      umma_commit(bar_s);
      issued = true;
    }
    // the next tile's rows stream in while this one computes (their buffer's last readers, the
    // MMAs of the previous tile, have completed)
    if (qt + 1 < n_qt) issue_q(qt + 1, buf ^ 1);
    cp_async_commit();
    // ---- teacher, index probabilities, dzI and KL: thread = key, its warpgroup's 8 positions
    if (mbar_wait(bar_s, nt & 1, abort, st, 0xA01)) {
      tc_fence_after();
      const int key = quad * 32 + lane;
      const int64_t j = j0 + key;
      const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
      uint32_t sx[2][32], zx[8];
      tmem_ld_x32(tmem + lane_base + kTS + half * 64, sx[0]);
      tmem_ld_x32(tmem + lane_base + kTS + half * 64 + 32, sx[1]);
      tmem_ld_x8(tmem + lane_base + kTZ + half * 8, zx);
      tmem_ld_wait();
      reg_fence32(sx[0]);
      reg_fence32(sx[1]);
      reg_fence8(zx);
      float dz[8], klv[8];
#pragma unroll
      for (int pl = 0; pl < 8; ++pl) {
        const int p = half * 8 + pl;
        const int32_t t = tpos_s[p];
        const bool valid = t >= 0 && j <= (int64_t)t;
        float ps = 0.f;
#pragma unroll
        for (int hd = 0; hd < 8; ++hd) {
          const int r = pl * 8 + hd;  // column within this warpgroup's 64
          ps += ex2_approx(fmaf(__uint_as_float(sx[r >> 5][r & 31]), sl2, -lse2_s[half * 64 + r]));
        }
        const float pbar = valid ? ps * 0.125f : 0.f;
        const float zl2 = fmaf(__uint_as_float(zx[pl]), sI2, -lseI2_s[p]);  // log2 pI
        const float pI = valid ? ex2_approx(zl2) : 0.f;
        dz[pl] = w_kl * (pI - pbar);
        klv[pl] = pbar > 0.f ? pbar * (wtc::lg2_approx(pbar) - zl2) * kLn2 : 0.f;
      }
      uint32_t pk[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) pk[u] = pack_bf16x2(dz[2 * u], dz[2 * u + 1]);
      wtc::tmem_st_x4(tmem + lane_base + kTDZ + half * 4, pk);
#pragma unroll
      for (int pl = 0; pl < 8; ++pl)
        *reinterpret_cast<uint16_t*>(sm + kDZ + off(half * 8 + pl, key, kChunk16)) =
            (uint16_t)(pack_bf16x2(dz[pl], 0.f) & 0xFFFFu);
#pragma unroll
      for (int pl = 0; pl < 8; ++pl) {
        float v = klv[pl];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) kl_s[warp][pl] = v;
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
    }
    __syncthreads();
    if (*abort) break;
    // ---- dk^I += dzI^T Q^I and dq^I^T = K^I^T dzI^T
    if (warp == 0 && lane == 0) {
      tc_fence_after();
      mma_bf16_ts(tmem + kTDK, tmem + kTDZ, umma_desc_mnmajor_sw128(qib, kChunk16), kIdescDK, nt > 0 ? 1u : 0u);
#pragma unroll
      for (int ks = 0; ks < kKeys / 16; ++ks) {
        const int c = ks >> 2, kk = ks & 3;
        mma_bf16_ss(tmem + kTDQ, umma_desc_mnmajor_sw128(sb + kKI + ks * 16 * 128, kChunk128),
                    umma_desc_kmajor(sb + kDZ + c * kChunk16 + kk * 32, 128), kIdescDQ, ks > 0);
      }
      umma_commit(bar_q);
    }
    if (tid < kPos) {  // the tile's KL sums: the four warps of the position's warpgroup
      const int h2 = tid >> 3, pl = tid & 7;
      const float v = kl_s[4 * h2][pl] + kl_s[4 * h2 + 1][pl] + kl_s[4 * h2 + 2][pl] + kl_s[4 * h2 + 3][pl];
      const int32_t t = tpos_s[tid];
      if (t >= 0 && v != 0.f) red_add(kl + (int64_t)g * N + t, v);
    }
    if (qt + 1 < n_qt) load_row_info(qt + 1);
    if (mbar_wait(bar_q, nt & 1, abort, st, 0xA02)) {
      tc_fence_after();
      // dq^I: thread = dim (TMEM lane), its warpgroup's 8 positions
      const int dim = quad * 32 + lane;
      uint32_t x[8];
      tmem_ld_x8(tmem + ((uint32_t)(quad * 32) << 16) + kTDQ + half * 8, x);
      tmem_ld_wait();
      reg_fence8(x);
#pragma unroll
      for (int pl = 0; pl < 8; ++pl) {
        const int32_t t = tpos_s[half * 8 + pl];
        if (t >= (int32_t)j0) red_add(dq_idx + ((int64_t)t * G + g) * DI + dim, sI * __uint_as_float(x[pl]));
      }
      tc_fence_before();
    }
    __syncthreads();
    if (*abort) break;
  }
  // ---- dk^I of the CTA's keys: thread = key, its warpgroup's 64 dims; the groups add up in dk_idx
  if (!*abort) {
    tc_fence_after();
    const int key = quad * 32 + lane;
    const int64_t j = j0 + key;
#pragma unroll 1
    for (int cc = 2 * half; cc < 2 * half + 2; ++cc) {
      uint32_t x[32];
      tmem_ld_x32(tmem + ((uint32_t)(quad * 32) << 16) + kTDK + cc * 32, x);
      tmem_ld_wait();
      if (j < N)
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          wtc::red_add4(dk_idx + j * DI + cc * 32 + e, sI * __uint_as_float(x[e]), sI * __uint_as_float(x[e + 1]),
                        sI * __uint_as_float(x[e + 2]), sI * __uint_as_float(x[e + 3]));
    }
    tc_fence_before();
  }
  cp_async_wait<0>();  // no copy of ours is left in flight when the CTA exits
  __syncthreads();
  if (warp == 0) {
    if (lane == 0 && *abort && issued) {  // let the MMAs in flight finish before TMEM is released
      umma_commit(bar_drain);
      mbar_wait(bar_drain, 0, nullptr, st, 0xAF1);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool warmup_tc_supported(int d, int d_I, int H_q, int H_kv) { return d == 128 && d_I == 128 && H_q == 8 * H_kv; }

cudaError_t launch_warmup_grad_tc(const void* q, const void* k, const void* q_idx, const void* k_idx, int64_t N,
                                  int H_q, int H_kv, float scale, float kl_weight, const float* lse, const float* lseI,
                                  float* dq_idx, float* dk_idx, float* kl, DeviceStatus* st, cudaStream_t s) {
  cudaError_t e;
  if ((e = cudaMemsetAsync(dq_idx, 0, (size_t)N * H_kv * 128 * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dk_idx, 0, (size_t)N * 128 * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(kl, 0, (size_t)H_kv * N * 4, s)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(warmup_grad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                wtc::kBytes)) != cudaSuccess)
    return e;
  const int64_t n_kt = (N + wtc::kKeys - 1) / wtc::kKeys;
  warmup_grad_tc_kernel<<<dim3((unsigned)H_kv, (unsigned)n_kt), wtc::kThreads, wtc::kBytes, s>>>(
      (const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)q_idx, (const uint16_t*)k_idx, lse, lseI, N, H_q,
      H_kv, scale, kl_weight, dq_idx, dk_idx, kl, st);
  return cudaGetLastError();
}

}  // namespace msa
