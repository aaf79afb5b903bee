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
// its positions, writes it (bf16) to TMEM (the A operand of dk^I) and to a
// K-major shared tile (the B operand of dq^I), and adds its KL terms;
//   dk^I  += dzI^T Q^I   (A from TMEM, Q^I as MN-major B), accumulated in
//                         TMEM over every query tile of the CTA and written
//                         once at the end;
//   dq^I^T = K^I^T dzI^T (K^I as MN-major A, M = d_I, N = 16 positions),
//                         added to dq^I with fp32 reductions (32 consecutive
//                         dims per warp instruction).
// Roles: a producer warp (TMA boxes of the query tiles' Q and Q^I into three
// slots, and each tile's lse row info), an MMA warp (one thread issues), and
// 16 softmax warps, 4 positions each.  They hand over through mbarriers:
// S^T, Z^T, dzI and dq^I^T have two TMEM buffers each, so S^T of tile n + 1
// runs on the tensor cores while tile n's exponentials do, and tile n's dk^I
// and dq^I products run while tile n + 1's do; a warp reads tile n's dq^I
// after its softmax of tile n + 1.  Barriers that a warp could reach again
// before the others leave them come in pairs (one per tile parity).  The main
// scores are computed once per (key, query) pair here; the forward pass keeps
// its own.
//
// Forward, query-outer: one CTA per (query tile of 16 positions x 8 heads,
// group), two CTAs per SM (256 TMEM columns and 96 KB each, so one CTA's MMAs
// run while the other's softmax does), heaviest tiles first.  Per 128-key
// tile: S = Q K^T into TMEM; both warpgroups take half of the key columns of
// every row (row maxima and sums exchanged through shared memory) and write P
// (bf16) back over their half of S; O += P V with P read from TMEM and V as
// an MN-major operand.  The running maximum is lazy: O and the row sum are
// rescaled only when a row's maximum grows by more than 2^8, so P stays below
// 256 and the rescale of O in TMEM is rare.  The next tile's K lands while
// the softmax runs, its V while the next S is computed.
// Index lse: one CTA per (128 positions, group), Z = Q^I K^I^T per 128-key
// tile into TMEM (two buffers), each thread keeps an exact online log-sum-exp
// of its row.
#include <math.h>

#include "msa_sm100.cuh"

namespace msa {

namespace {

using namespace sm100;

namespace wtc {
constexpr int kKeys = 128;   // keys of a CTA
constexpr int kPos = 16;     // positions of a query tile
constexpr int kRows = 128;   // 16 positions x 8 heads
constexpr int kSoftWarps = 16;                  // four warpgroups, 4 positions each
constexpr int kWarpLoad = 16, kWarpMma = 17;    // producer (TMA, row info) and MMA issuer
constexpr int kThreads = 32 * (kSoftWarps + 2);
constexpr int kSlots = 3;                       // query tiles in flight (Q, Q^I, row info)
constexpr int kChunk128 = 128 * 128;  // one 64-column chunk of a 128-row bf16 tile, bytes
constexpr int kTile128 = 2 * kChunk128;
constexpr int kChunk16 = 16 * 128;    // one 64-column chunk of a 16-row bf16 tile
constexpr int kTile16 = 2 * kChunk16;
constexpr int kK = 0, kKI = kTile128, kQ = 2 * kTile128;  // Q: kSlots buffers
constexpr int kQI = kQ + kSlots * kTile128;                 // Q^I: kSlots buffers
constexpr int kDZ = kQI + kSlots * kTile16;                 // dzI [16 positions][128 keys], K-major: two buffers
constexpr int kBar = kDZ + 2 * kTile16;
constexpr int kNumBars = 18;
constexpr int kBytes = 1024 + kBar + 8 * kNumBars;
constexpr uint32_t kTileTx = kTile128 + kTile16;  // bytes of one query tile's Q and Q^I
// TMEM columns: S^T, Z^T, dq^I^T and dzI^T (A operand, bf16 packed) with two buffers each, dk^I.
// Softmax warp w (TMEM lanes 32 (w % 4) ..) owns positions 4 (w / 4) .. + 3 of a query tile.
constexpr uint32_t kTS = 0, kTZ = 256, kTDQ = 288, kTDZ = 320, kTDK = 384;
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128);
constexpr uint32_t kIdescZ = idesc_bf16_f32(128, 16);
constexpr uint32_t kIdescDK = idesc_bf16_f32(128, 128) | (1u << 16);  // B MN-major
constexpr uint32_t kIdescDQ = idesc_bf16_f32(128, 16) | (1u << 15);   // A MN-major
// Byte offset of element (row r, column c) of a 128B-swizzled K-major bf16
// tile whose 64-column chunks are `chunk` bytes apart (8-row groups 1 KB apart):
// the layout a TMA box of 64 columns lands in, one box per chunk.
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
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
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
__device__ __forceinline__ void tmem_ld_x4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
__device__ __forceinline__ void reg_fence4(uint32_t (&r)[4]) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]));
}
__device__ __forceinline__ void tmem_st_x2(uint32_t taddr, const uint32_t (&r)[2]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1,%2};\n" ::"r"(taddr), "r"(r[0]), "r"(r[1])
               : "memory");
}
// A bounded wait whose result every lane of the warp shares (warp-collective work follows it).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, DeviceStatus* st,
                                          unsigned code) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, st, code, 64));
}
}  // namespace wtc

__global__ void __launch_bounds__(wtc::kThreads, 1) warmup_grad_tc_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qi,
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_ki,
    const float* __restrict__ lse, const float* __restrict__ lseI, int64_t N, int G, float scale, float w_kl,
    float* __restrict__ dq_idx, float* __restrict__ dk_idx, float* __restrict__ kl, DeviceStatus* st) {
  using namespace wtc;
  constexpr int DI = 128;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ __align__(16) float lse2_s[kSlots][kRows];   // main lse of each tile row, log2 units
  __shared__ float lseI2_s[kSlots][kPos];   // lse^I of each position, log2 units
  __shared__ int32_t tpos_s[kSlots][kPos];  // position of each tile position, -1 past N
  const uint32_t bar = sb + kBar;
  const uint32_t kv_full = bar;
  auto full = [&](int i) { return bar + 8u * (1 + i); };     // producer -> MMA, softmax (count 32 + tx)
  auto empty = [&](int i) { return bar + 8u * (4 + i); };    // softmax -> producer (count 8)
  auto s_full = [&](int i) { return bar + 8u * (7 + i); };   // MMA -> softmax (commit)
  auto s_empty = [&](int i) { return bar + 8u * (9 + i); };  // softmax -> MMA (count 8)
  // Per buffer parity, so that no warp can reach a barrier's next use before every arrival of this one:
  auto dz_full = [&](int i) { return bar + 8u * (11 + i); };  // softmax -> MMA (count 8): dzI of tile written
  auto q_done = [&](int i) { return bar + 8u * (13 + i); };   // MMA -> softmax (commit): dk^I, dq^I done
  auto dq_read = [&](int i) { return bar + 8u * (15 + i); };  // softmax -> MMA (count 8): dq buffer i read
  const uint32_t drain = bar + 8u * 17;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = (int)(blockIdx.x % (unsigned)G);
  const int64_t j0 = (int64_t)(blockIdx.x / (unsigned)G) * kKeys;  // launch order: the heaviest key tiles first
  const int64_t n_qt = (N + kPos - 1) / kPos;
  const int64_t qt0 = j0 / kPos;  // the first query tile with a position >= j0
  const int n_tiles = (int)(n_qt - qt0);
  if (tid == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(full(i), 32);
      mbar_init(empty(i), kSoftWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full(i), 1);
      mbar_init(s_empty(i), kSoftWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(dz_full(i), kSoftWarps);
      mbar_init(q_done(i), 1);
      mbar_init(dq_read(i), kSoftWarps);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&tmem_slot), 512);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;
  const float kLog2e = 1.4426950408889634f;

  if (warp == kWarpLoad) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_qi);
      mbar_arrive_expect_tx(kv_full, (uint32_t)(2 * kTile128));
      for (int c = 0; c < 2; ++c) {
        tma_load_3d(sb + kK + c * kChunk128, &tm_k, c * 64, g, (int32_t)j0, kv_full);
        tma_load_3d(sb + kKI + c * kChunk128, &tm_ki, c * 64, 0, (int32_t)j0, kv_full);
      }
    }
    int issued = 0;
    for (int n = 0; n < n_tiles; ++n) {
      const int slot = n % kSlots;
      if (n >= kSlots && !warp_wait(empty(slot), (uint32_t)((n / kSlots - 1) & 1), abort, st, 0xA10)) break;
      const int64_t t0 = (qt0 + n) * kPos;
      // row info: lse of rows 8 p + h (coalesced along p), and lse^I and the position of each p
#pragma unroll
      for (int m = 0; m < kRows / 32; ++m) {
        const int idx = lane + 32 * m, h = idx >> 4, p = idx & 15;
        const int64_t t = t0 + p;
        lse2_s[slot][p * 8 + h] = t < N ? __ldg(lse + ((int64_t)g * 8 + h) * N + t) * kLog2e : 0.f;
      }
      if (lane < kPos) {
        const int64_t t = t0 + lane;
        tpos_s[slot][lane] = t < N ? (int32_t)t : -1;
        lseI2_s[slot][lane] = t < N ? __ldg(lseI + (int64_t)g * N + t) * kLog2e : 0.f;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(full(slot), kTileTx);
        for (int c = 0; c < 2; ++c) {
          tma_load_3d(sb + kQ + slot * kTile128 + c * kChunk128, &tm_q, c * 64, g * 8, (int32_t)t0, full(slot));
          tma_load_3d(sb + kQI + slot * kTile16 + c * kChunk16, &tm_qi, c * 64, g, (int32_t)t0, full(slot));
        }
      } else {
        mbar_arrive(full(slot));
      }
      issued = n + 1;
    }
    // after an abort: the copies still in flight land before the CTA exits
    if (*abort && lane == 0)
      for (int n = max(0, issued - kSlots); n < issued; ++n)
        mbar_wait(full(n % kSlots), (uint32_t)((n / kSlots) & 1), nullptr, st, 0xAF2);
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------------- MMA issuer
    bool ok = warp_wait(kv_full, 0, abort, st, 0xA20);
    bool issued = false;
    for (int n = 0; ok && n <= n_tiles; ++n) {
      if (n < n_tiles) {  // S^T(n), Z^T(n) into TMEM buffer n % 2
        const int slot = n % kSlots, b = n & 1;
        if (!(ok = warp_wait(full(slot), (uint32_t)((n / kSlots) & 1), abort, st, 0xA21))) break;
        if (n >= 2 && !(ok = warp_wait(s_empty(b), (uint32_t)((n / 2 - 1) & 1), abort, st, 0xA22))) break;
        if (lane == 0) {
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const int c = ks >> 2, kk = ks & 3;
            mma_bf16_ss(tmem + kTS + b * 128, umma_desc_kmajor(sb + kK + c * kChunk128 + kk * 32, 128),
                        umma_desc_kmajor(sb + kQ + slot * kTile128 + c * kChunk128 + kk * 32, 128), kIdescS, ks > 0);
            mma_bf16_ss(tmem + kTZ + b * 16, umma_desc_kmajor(sb + kKI + c * kChunk128 + kk * 32, 128),
                        umma_desc_kmajor(sb + kQI + slot * kTile16 + c * kChunk16 + kk * 32, 128), kIdescZ, ks > 0);
          }
          umma_commit(s_full(b));
        }
        issued = true;
      }
      if (n >= 1) {  // dk^I += dzI^T Q^I and dq^I^T = K^I^T dzI^T of tile m = n - 1 (buffers m % 2)
        const int m = n - 1, slot = m % kSlots, bm = m & 1;
        if (!(ok = warp_wait(dz_full(bm), (uint32_t)((m / 2) & 1), abort, st, 0xA23))) break;
        if (m >= 2 && !(ok = warp_wait(dq_read(bm), (uint32_t)((m / 2 - 1) & 1), abort, st, 0xA24))) break;
        if (lane == 0) {
          tc_fence_after();
          mma_bf16_ts(tmem + kTDK, tmem + kTDZ + bm * 8,
                      umma_desc_mnmajor_sw128(sb + kQI + slot * kTile16, kChunk16), kIdescDK, m > 0 ? 1u : 0u);
#pragma unroll
          for (int ks = 0; ks < kKeys / 16; ++ks) {
            const int c = ks >> 2, kk = ks & 3;
            mma_bf16_ss(tmem + kTDQ + bm * 16, umma_desc_mnmajor_sw128(sb + kKI + ks * 16 * 128, kChunk128),
                        umma_desc_kmajor(sb + kDZ + bm * kTile16 + c * kChunk16 + kk * 32, 128), kIdescDQ, ks > 0);
          }
          umma_commit(q_done(bm));
        }
      }
    }
    if (!ok && issued && lane == 0) {  // let the MMAs in flight finish before TMEM is released
      umma_commit(drain);
      mbar_wait(drain, 0, nullptr, st, 0xAF1);
    }
  } else {
    // ---------------------------------------------------------------- softmax warps: thread = key
    const int quad = warp & 3, qtr = warp >> 2;  // TMEM lane quadrant; positions 4 qtr .. 4 qtr + 3
    const int key = quad * 32 + lane;
    const int64_t j = j0 + key;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const float sl2 = scale * kLog2e;  // main scores -> log2 units
    const float sI = 1.0f / sqrtf((float)DI);
    const float sI2 = sI * kLog2e;     // index logits -> log2 units
    const float kLn2 = 0.69314718055994530942f;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    bool ok = true;
    // iteration n: the softmax of tile n, then the dq^I of tile n - 1 (whose products ran meanwhile)
    for (int n = 0; n <= n_tiles; ++n) {
      if (n < n_tiles) {
        const int b = n & 1, slot = n % kSlots;
        if (!(ok = warp_wait(s_full(b), (uint32_t)((n / 2) & 1), abort, st, 0xA30))) break;
        if (!(ok = warp_wait(full(slot), (uint32_t)((n / kSlots) & 1), abort, st, 0xA31))) break;
        tc_fence_after();
        uint32_t sx[32], zx[4];
        tmem_ld_x32(tmem + lane_base + kTS + b * 128 + qtr * 32, sx);
        tmem_ld_x4(tmem + lane_base + kTZ + b * 16 + qtr * 4, zx);
        tmem_ld_wait();
        reg_fence32(sx);
        reg_fence4(zx);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty(b));  // the MMA may overwrite this S^T / Z^T buffer
        float dz[4], klv[4];
        const float2* lse2p = reinterpret_cast<const float2*>(&lse2_s[slot][qtr * 32]);
#pragma unroll
        for (int pl = 0; pl < 4; ++pl) {
          const int p = qtr * 4 + pl;
          const int32_t t = tpos_s[slot][p];
          const bool valid = t >= 0 && j <= (int64_t)t;
          float ps = 0.f;
#pragma unroll
          for (int hd = 0; hd < 8; hd += 2) {
            const int r = pl * 8 + hd;  // column within this warpgroup's 32
            const float2 l2 = lse2p[r >> 1];
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sx[r]), __uint_as_float(sx[r + 1])), sl2x2, f2_pack(-l2.x, -l2.y)),
                      a0, a1);
            ps += ex2_approx(a0) + ex2_approx(a1);
          }
          const float pbar = valid ? ps * 0.125f : 0.f;
          const float zl2 = fmaf(__uint_as_float(zx[pl]), sI2, -lseI2_s[slot][p]);  // log2 pI
          const float pI = valid ? ex2_approx(zl2) : 0.f;
          dz[pl] = w_kl * (pI - pbar);
          klv[pl] = pbar > 0.f ? pbar * (lg2_approx(pbar) - zl2) * kLn2 : 0.f;
        }
        // dzI to TMEM (A of dk^I) and to the K-major shared tile (B of dq^I), buffer n % 2; their last
        // readers, the products of tile n - 2, completed before this warp read that tile's dq^I
        const uint32_t pk[2] = {pack_bf16x2(dz[0], dz[1]), pack_bf16x2(dz[2], dz[3])};
        tmem_st_x2(tmem + lane_base + kTDZ + b * 8 + qtr * 2, pk);
#pragma unroll
        for (int pl = 0; pl < 4; ++pl)
          *reinterpret_cast<uint16_t*>(sm + kDZ + b * kTile16 + off(qtr * 4 + pl, key, kChunk16)) =
              (uint16_t)(pack_bf16x2(dz[pl], 0.f) & 0xFFFFu);
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dz_full(b));
        // this warp's KL sums over its 32 keys, one reduction per position
#pragma unroll
        for (int pl = 0; pl < 4; ++pl) {
          float v = klv[pl];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          const int32_t t = tpos_s[slot][qtr * 4 + pl];
          if (lane == 0 && t >= 0 && v != 0.f) red_add(kl + (int64_t)g * N + t, v);
        }
      }
      if (n >= 1) {  // dq^I of tile m = n - 1: thread = dim (TMEM lane), its warpgroup's 4 positions
        const int m = n - 1, bm = m & 1, slot = m % kSlots;
        if (!(ok = warp_wait(q_done(bm), (uint32_t)((m / 2) & 1), abort, st, 0xA32))) break;
        tc_fence_after();
        uint32_t x[4];
        tmem_ld_x4(tmem + lane_base + kTDQ + bm * 16 + qtr * 4, x);
        tmem_ld_wait();
        reg_fence4(x);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dq_read(bm));  // the product of tile m + 2 may overwrite these columns
#pragma unroll
        for (int pl = 0; pl < 4; ++pl) {
          const int32_t t = tpos_s[slot][qtr * 4 + pl];
          if (t >= 0) red_add(dq_idx + ((int64_t)t * G + g) * DI + key, sI * __uint_as_float(x[pl]));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(slot));  // tile m's Q, Q^I and row info are no longer read
      }
    }
    // dk^I of the CTA's keys: thread = key, its warpgroup's 32 dims; the groups add up in dk_idx
    if (ok && n_tiles > 0) {
      tc_fence_after();
      uint32_t x[32];
      tmem_ld_x32(tmem + lane_base + kTDK + qtr * 32, x);
      tmem_ld_wait();
      if (j < N)
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          red_add4(dk_idx + j * DI + qtr * 32 + e, sI * __uint_as_float(x[e]), sI * __uint_as_float(x[e + 1]),
                   sI * __uint_as_float(x[e + 2]), sI * __uint_as_float(x[e + 3]));
      tc_fence_before();
    }
  }
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

namespace wtf {
constexpr int kThreads = 256;
constexpr int kQ = 0, kK = wtc::kTile128, kV = 2 * wtc::kTile128;  // one 128 x 128 tile each
constexpr int kBar = 3 * wtc::kTile128;
constexpr int kBytes = 1024 + kBar + 64;
constexpr uint32_t kTS = 0, kTO = 128, kCols = 256;
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128) | (1u << 16);  // V as MN-major B
constexpr float kLazy = 8.0f;  // log2 units a row maximum may grow before O is rescaled
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
}  // namespace wtf

__global__ void __launch_bounds__(wtf::kThreads, 2) warmup_fwd_tc_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ kc, const uint16_t* __restrict__ vc, int64_t N,
    int H_q, int G, float scale, uint16_t* __restrict__ out, float* __restrict__ lse, DeviceStatus* st) {
  using namespace wtf;
  using wtc::kChunk128;
  using wtc::off;
  constexpr int D = 128;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ float ex_m[2][128], ex_l[2][128];  // the two halves' row maxima and sums
  const uint32_t bar_s = sb + kBar, bar_o = sb + kBar + 8, bar_drain = sb + kBar + 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;  // TMEM lane quadrant; key columns 64 half .. + 63
  const int g = (int)(blockIdx.x % (unsigned)G);
  const int64_t n_qt = (N + wtc::kPos - 1) / wtc::kPos;
  const int64_t t0 = (n_qt - 1 - (int64_t)(blockIdx.x / (unsigned)G)) * wtc::kPos;  // the longest rows first
  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    mbar_init(bar_drain, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), kCols);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;
  const float sl2 = scale * 1.4426950408889634f;  // scores -> log2 units
  const int64_t kv_row = (int64_t)G * D;
  // Q rows r = 8 p + h: position t0 + p, head g*8 + h
#pragma unroll
  for (int m = 0; m < wtc::kRows * 16 / kThreads; ++m) {
    const int i = tid + m * kThreads;
    const int r = i >> 4, c = (i & 15) * 8;
    const int64_t t = t0 + (r >> 3);
    const bool ok = t < N;
    cp_async_16(sm + kQ + off(r, c, kChunk128), ok ? q + (t * H_q + (int64_t)g * 8 + (r & 7)) * D + c : q,
                ok ? 16 : 0);
  }
  // keys [128 i, 128 i + 128) of group g into the K or V tile
  auto load_kv = [&](int base, const uint16_t* src, int64_t i) {
#pragma unroll
    for (int m = 0; m < 128 * 16 / kThreads; ++m) {
      const int e = tid + m * kThreads;
      const int r = e >> 4, c = (e & 15) * 8;
      const int64_t j = i * 128 + r;
      const bool ok = j < N;
      cp_async_16(sm + base + off(r, c, kChunk128), ok ? src + j * kv_row + (int64_t)g * D + c : src, ok ? 16 : 0);
    }
  };
  const int64_t t_last = min(t0 + wtc::kPos, N) - 1;  // keys [0, t_last] are visible to some row
  const int64_t n_kv = t_last / 128 + 1;
  load_kv(kK, kc, 0);
  load_kv(kV, vc, 0);
  cp_async_commit();
  const int row = quad * 32 + lane;
  const int64_t t = t0 + (row >> 3);  // this thread's row
  const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
  const uint32_t scol = tmem + lane_base + kTS + half * 64;
  const uint32_t ocol = tmem + lane_base + kTO + half * 64;
  float m_used = __int_as_float(0xff800000);  // the row's maximum in use (log2 units)
  float l_run = 0.f;
  bool issued = false;
  for (int64_t i = 0; i < n_kv; ++i) {
    cp_async_wait<0>();  // K(i) and V(i) (and, at i = 0, Q)
    fence_proxy_async_smem();
    __syncthreads();
    if (warp == 0 && lane == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int c = ks >> 2, kk = ks & 3;
        mma_bf16_ss(tmem + kTS, umma_desc_kmajor(sb + kQ + c * kChunk128 + kk * 32, 128),
                    umma_desc_kmajor(sb + kK + c * kChunk128 + kk * 32, 128), kIdescS, ks > 0);
      }
      umma_commit(bar_s);
      issued = true;
    }
    // every thread takes the same branch (the TMEM loads below are warp-collective)
    const bool ok_s = __syncthreads_and(mbar_wait(bar_s, (uint32_t)(i & 1), abort, st, 0xB01));
    // S(i) is done, and so is P V(i - 1) (issued before it): K is free for the next tile
    if (i + 1 < n_kv) load_kv(kK, kc, i + 1);
    cp_async_commit();
    if (ok_s) {
      tc_fence_after();
      const int64_t key0 = i * 128 + half * 64;
      // last visible column of this half for this row (-1: none); rows past N see nothing
      const int lim = t < N ? (int)max((int64_t)-1, min((int64_t)63, t - key0)) : -1;
      uint32_t x[2][32];
      tmem_ld_x32(scol, x[0]);
      tmem_ld_x32(scol + 32, x[1]);
      tmem_ld_wait();
      reg_fence32(x[0]);
      reg_fence32(x[1]);
      // tiles below the diagonal for every row of the warp take the unmasked path
      const bool full = __all_sync(0xffffffffu, lim == 63);
      float mx = __int_as_float(0xff800000);
      if (full) {
        float m2[2];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          m2[cc] = __int_as_float(0xff800000);
#pragma unroll
          for (int e = 0; e < 32; e += 2) m2[cc] = max3(m2[cc], __uint_as_float(x[cc][e]), __uint_as_float(x[cc][e + 1]));
        }
        mx = fmaxf(m2[0], m2[1]);
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (e <= lim) mx = fmaxf(mx, __uint_as_float(x[e >> 5][e & 31]));
      }
      ex_m[half][row] = mx;
      __syncthreads();
      const float mt = fmaxf(ex_m[0][row], ex_m[1][row]);
      const float mt2 = mt == __int_as_float(0xff800000) ? mt : mt * sl2;
      // both halves take the same decision for the row: the maximum in use moves only past 2^8 of growth
      const bool rescale = mt2 > m_used + kLazy;
      const float alpha = !rescale || m_used == __int_as_float(0xff800000) ? 0.f : ex2_approx(m_used - mt2);
      if (rescale) {
        l_run *= alpha;
        m_used = mt2;
      }
      float ls = 0.f;
      if (full) {
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nm2 = f2_pack(-m_used, -m_used);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {  // 32 keys at a time -> 16 packed columns
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float a0, a1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(x[cc][e]), __uint_as_float(x[cc][e + 1])), sl2x2,
                                       nm2),
                           a0, a1);
            a0 = ex2_approx(a0);
            a1 = ex2_approx(a1);
            ls += a0 + a1;
            pk[e >> 1] = pack_bf16x2(a0, a1);
          }
          tmem_st_x16(scol + cc * 16, pk);  // keys of this half -> its first 32 columns, packed
        }
      } else {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int c0 = cc * 32 + e;
            const float p0 = c0 <= lim ? ex2_approx(fmaf(__uint_as_float(x[cc][e]), sl2, -m_used)) : 0.f;
            const float p1 = c0 + 1 <= lim ? ex2_approx(fmaf(__uint_as_float(x[cc][e + 1]), sl2, -m_used)) : 0.f;
            ls += p0 + p1;
            pk[e >> 1] = pack_bf16x2(p0, p1);
          }
          tmem_st_x16(scol + cc * 16, pk);
        }
      }
      if (rescale && i > 0) {  // O holds P V of earlier tiles (complete: see above); rescale this half's columns
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t o[32];
          tmem_ld_x32(ocol + cc * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          wtf::tmem_st_x32(ocol + cc * 32, o);
        }
      }
      ex_l[half][row] = ls;
      tmem_st_wait();
      tc_fence_before();
    }
    __syncthreads();
    if (*abort) break;
    l_run += ex_l[0][row] + ex_l[1][row];
    if (warp == 0 && lane == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {  // keys 16 ks ..: half ks / 4, packed at column 64 half + 8 (ks % 4)
        const uint32_t acol = tmem + kTS + (uint32_t)(64 * (ks >> 2) + 8 * (ks & 3));
        mma_bf16_ts(tmem + kTO, acol, umma_desc_mnmajor_sw128(sb + kV + ks * 16 * 128, kChunk128), kIdescPV,
                    (i > 0 || ks > 0) ? 1u : 0u);
      }
      umma_commit(bar_o);
    }
    if (!__syncthreads_and(mbar_wait(bar_o, (uint32_t)(i & 1), abort, st, 0xB02))) break;
    // P V(i) is done: V is free for the next tile (its S runs while V lands)
    if (i + 1 < n_kv) load_kv(kV, vc, i + 1);
    cp_async_commit();
  }
  // ---- out = O / l and lse: thread = row, its half's 64 columns
  if (!*abort) {
    tc_fence_after();
    uint32_t o[2][32];
    tmem_ld_x32(ocol, o[0]);
    tmem_ld_x32(ocol + 32, o[1]);
    tmem_ld_wait();
    if (t < N) {
      const float il = l_run > 0.f ? 1.f / l_run : 0.f;
      uint16_t* orow = out + (t * H_q + (int64_t)g * 8 + (row & 7)) * D + half * 64;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint4 v;
        v.x = pack_bf16x2(__uint_as_float(o[u >> 2][(u & 3) * 8 + 0]) * il, __uint_as_float(o[u >> 2][(u & 3) * 8 + 1]) * il);
        v.y = pack_bf16x2(__uint_as_float(o[u >> 2][(u & 3) * 8 + 2]) * il, __uint_as_float(o[u >> 2][(u & 3) * 8 + 3]) * il);
        v.z = pack_bf16x2(__uint_as_float(o[u >> 2][(u & 3) * 8 + 4]) * il, __uint_as_float(o[u >> 2][(u & 3) * 8 + 5]) * il);
        v.w = pack_bf16x2(__uint_as_float(o[u >> 2][(u & 3) * 8 + 6]) * il, __uint_as_float(o[u >> 2][(u & 3) * 8 + 7]) * il);
        *reinterpret_cast<uint4*>(orow + u * 8) = v;
      }
      if (half == 0)
        lse[((int64_t)g * 8 + (row & 7)) * N + t] =
            l_run > 0.f ? (m_used + __log2f(l_run)) * 0.69314718055994530942f : __int_as_float(0xff800000);
    }
    tc_fence_before();
  }
  cp_async_wait<0>();
  __syncthreads();
  if (warp == 0) {
    if (lane == 0 && *abort && issued) {
      umma_commit(bar_drain);
      mbar_wait(bar_drain, 0, nullptr, st, 0xBF1);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

// ---- the index branch's log-sum-exp over j <= t: thread = position
namespace wti {
constexpr int kThreads = 128;
constexpr int kQI = 0, kKI = wtc::kTile128;  // K^I: two buffers
constexpr int kBar = 3 * wtc::kTile128;
constexpr int kBytes = 1024 + kBar + 64;
constexpr uint32_t kCols = 256;
constexpr uint32_t kIdesc = idesc_bf16_f32(128, 128);
}  // namespace wti

__global__ void __launch_bounds__(wti::kThreads, 2) warmup_index_lse_tc_kernel(
    const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ k_idx, int64_t N, int G,
    float* __restrict__ lseI, DeviceStatus* st) {
  using namespace wti;
  using wtc::kChunk128;
  using wtc::off;
  constexpr int DI = 128;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  const uint32_t bar0 = sb + kBar, bar_drain = sb + kBar + 16;  // bar0 + 8 b: Z buffer b complete
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = (int)(blockIdx.x % (unsigned)G);
  const int64_t n_pt = (N + 127) / 128;
  const int64_t p0 = (n_pt - 1 - (int64_t)(blockIdx.x / (unsigned)G)) * 128;  // the longest rows first
  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    mbar_init(bar_drain, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), kCols);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;
  const float sI2 = 1.4426950408889634f / sqrtf((float)DI);
  for (int e = tid; e < 128 * 16; e += kThreads) {
    const int r = e >> 4, c = (e & 15) * 8;
    const int64_t t = p0 + r;
    const bool ok = t < N;
    cp_async_16(sm + kQI + off(r, c, kChunk128), ok ? q_idx + (t * G + g) * DI + c : q_idx, ok ? 16 : 0);
  }
  auto load_k = [&](int b, int64_t i) {
    for (int e = tid; e < 128 * 16; e += kThreads) {
      const int r = e >> 4, c = (e & 15) * 8;
      const int64_t j = i * 128 + r;
      const bool ok = j < N;
      cp_async_16(sm + kKI + b * wtc::kTile128 + off(r, c, kChunk128), ok ? k_idx + j * DI + c : k_idx,
                  ok ? 16 : 0);
    }
  };
  const int64_t t_last = min(p0 + 128, N) - 1;
  const int64_t n_kt = t_last / 128 + 1;
  load_k(0, 0);
  cp_async_commit();
  const int64_t t = p0 + warp * 32 + lane;  // this thread's position (TMEM lane)
  float m = __int_as_float(0xff800000), l = 0.f;
  bool issued = false;
  for (int64_t i = 0; i < n_kt; ++i) {
    const int b = (int)(i & 1);
    if (i + 1 < n_kt) load_k(b ^ 1, i + 1);  // that buffer's last MMA (tile i - 1) completed
    cp_async_commit();
    cp_async_wait<1>();  // tile i's keys (and Q^I)
    fence_proxy_async_smem();
    __syncthreads();
    if (warp == 0 && lane == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < DI / 16; ++ks) {
        const int c = ks >> 2, kk = ks & 3;
        mma_bf16_ss(tmem + (uint32_t)(b * 128), umma_desc_kmajor(sb + kQI + c * kChunk128 + kk * 32, 128),
                    umma_desc_kmajor(sb + kKI + b * wtc::kTile128 + c * kChunk128 + kk * 32, 128), kIdesc, ks > 0);
      }
      umma_commit(bar0 + 8 * b);
      issued = true;
    }
    if (!__syncthreads_and(mbar_wait(bar0 + 8 * b, (uint32_t)((i >> 1) & 1), abort, st, 0xC01))) break;
    tc_fence_after();
    const int lim = t < N ? (int)max((int64_t)-1, min((int64_t)127, t - i * 128)) : -1;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t x[32];
      tmem_ld_x32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(b * 128 + cc * 32), x);
      tmem_ld_wait();
      float mx = __int_as_float(0xff800000);
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (cc * 32 + e <= lim) mx = fmaxf(mx, __uint_as_float(x[e]) * sI2);
      if (mx == __int_as_float(0xff800000)) continue;
      const float mn = fmaxf(m, mx);
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (cc * 32 + e <= lim) s += ex2_approx(fmaf(__uint_as_float(x[e]), sI2, -mn));
      l = l * ex2_approx(m - mn) + s;  // 2^(-inf) = 0 at the first key
      m = mn;
    }
    tc_fence_before();
    __syncthreads();  // buffer b is read: the tile after next may overwrite it
  }
  if (!*abort && t < N)
    lseI[(int64_t)g * N + t] = l > 0.f ? (m + __log2f(l)) * 0.69314718055994530942f : __int_as_float(0xff800000);
  cp_async_wait<0>();
  __syncthreads();
  if (warp == 0) {
    if (lane == 0 && *abort && issued) {
      umma_commit(bar_drain);
      mbar_wait(bar_drain, 0, nullptr, st, 0xCF1);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kCols);
  }
}

}  // namespace

bool warmup_tc_supported(int d, int d_I, int H_q, int H_kv) { return d == 128 && d_I == 128 && H_q == 8 * H_kv; }

cudaError_t launch_warmup_fwd_tc(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                                 int64_t N, int H_q, int H_kv, float scale, void* out, float* lse, float* lseI,
                                 DeviceStatus* st, cudaStream_t s) {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(warmup_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, wtf::kBytes)) !=
      cudaSuccess)
    return e;
  const int64_t n_qt = (N + wtc::kPos - 1) / wtc::kPos;
  warmup_fwd_tc_kernel<<<(unsigned)(n_qt * H_kv), wtf::kThreads, wtf::kBytes, s>>>(
      (const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)v, N, H_q, H_kv, scale, (uint16_t*)out, lse, st);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(warmup_index_lse_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                wti::kBytes)) != cudaSuccess)
    return e;
  const int64_t n_pt = (N + 127) / 128;
  warmup_index_lse_tc_kernel<<<(unsigned)(n_pt * H_kv), wti::kThreads, wti::kBytes, s>>>(
      (const uint16_t*)q_idx, (const uint16_t*)k_idx, N, H_kv, lseI, st);
  return cudaGetLastError();
}

cudaError_t launch_warmup_grad_tc(const void* q, const void* k, const void* q_idx, const void* k_idx, int64_t N,
                                  int H_q, int H_kv, float scale, float kl_weight, const float* lse, const float* lseI,
                                  float* dq_idx, float* dk_idx, float* kl, DeviceStatus* st, cudaStream_t s) {
  constexpr int D = 128, DI = 128;
  alignas(64) unsigned char tq[128], tqi[128], tk[128], tki[128];
  // q [N][H_q][d] as boxes {64 dims, 8 heads, 16 positions}; q^I [N][G][d_I] as {64, 1, 16};
  // k [N][H_kv][d] as {64, 1, 128 keys}; k^I [N][d_I] as {64, 1, 128}: each box lands as one 64-column chunk
  // of the kernels' 128B-swizzled K-major tiles
  if (!encode_tmap_3d(tq, q, D, (uint64_t)H_q, (uint64_t)N, D * 2, (uint64_t)H_q * D * 2, 64, 8, 16, 128) ||
      !encode_tmap_3d(tqi, q_idx, DI, (uint64_t)H_kv, (uint64_t)N, DI * 2, (uint64_t)H_kv * DI * 2, 64, 1, 16, 128) ||
      !encode_tmap_3d(tk, k, D, (uint64_t)H_kv, (uint64_t)N, D * 2, (uint64_t)H_kv * D * 2, 64, 1, 128, 128) ||
      !encode_tmap_3d(tki, k_idx, DI, 1, (uint64_t)N, DI * 2, DI * 2, 64, 1, 128, 128))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if ((e = cudaMemsetAsync(dq_idx, 0, (size_t)N * H_kv * DI * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dk_idx, 0, (size_t)N * DI * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(kl, 0, (size_t)H_kv * N * 4, s)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(warmup_grad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                wtc::kBytes)) != cudaSuccess)
    return e;
  (void)H_q;
  const int64_t n_kt = (N + wtc::kKeys - 1) / wtc::kKeys;
  warmup_grad_tc_kernel<<<(unsigned)(n_kt * H_kv), wtc::kThreads, wtc::kBytes, s>>>(
      *reinterpret_cast<const CUtensorMap*>(tq), *reinterpret_cast<const CUtensorMap*>(tqi),
      *reinterpret_cast<const CUtensorMap*>(tk), *reinterpret_cast<const CUtensorMap*>(tki), lse, lseI, N, H_kv,
      scale, kl_weight, dq_idx, dk_idx, kl, st);
  return cudaGetLastError();
}

}  // namespace msa
