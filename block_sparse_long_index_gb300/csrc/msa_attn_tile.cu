// KV-outer attention tiles on the 5th-generation tensor cores.
//
// "MSA" study note 3-3 "Main Branch" (exact softmax over the selected
// support, per-head weights, group-shared blocks) and 3-5 (KV-outer:
// the queries that chose a KV block are concatenated into one large MMA that
// reuses the block from on-chip memory; hot blocks pre-chunked into tiles).
//
// A tile is (group g, block b, up to P = 128/gs query positions that chose b)
// and its 128 rows are (position, head of g).  Per tile:
//   S = Q K_b^T (128 x Bk fp32 in TMEM), causal mask j <= t, row softmax,
//   P (bf16, written back into S's TMEM columns), O = P V_b (128 x d fp32 in
//   TMEM, P read from TMEM as the A operand), then the normalised partial O
//   (bf16) and partial lse of every (t, slot, h) row.
// Roles (448 threads):
//   warps 0..3   Q loaders: loader w gathers the Q rows of tiles i = w mod 4
//                into Q buffer w with cp.async (128B-swizzled K-major layout),
//                so four tiles' gathers are in flight;
//   warp 4       TMEM owner; lane 0 issues tcgen05.mma: S(i+1) then PV(i)
//                (PV(i) first when tile i+1 needs another K/V block);
//   warps 5..12  two softmax warpgroups, one per tile parity, each with its own
//                S/P and O columns in TMEM: softmax(i) then epilogue(i);
//   warp 13      K/V loader: one TMA load of K_b and V_b per run of tiles of
//                the same block, released by the MMA issuer after the run's
//                last P V.
// K_b and Q feed the tensor cores as K-major shared-memory operands, V_b as an
// MN-major one (d contiguous), P from TMEM.  Every wait is bounded; on expiry
// the kernel flags a timeout, drains its own async work and exits.
#include <math.h>

#include "msa_sm100.cuh"

namespace msa {

namespace {

using namespace sm100;

constexpr int kRowsT = 128;
constexpr int kQLoaders = 4;
constexpr int kWarpMma = 4;
constexpr int kWarpSoft0 = 5;
constexpr int kWarpKv = 13;
constexpr int kThreadsT = 14 * 32;
constexpr int kSoftWarps = 4;  // per warpgroup

template <int D, int BK>
struct AttnLayout {
  static constexpr int NCD = D / 64;  // 64-column chunks of d
  static constexpr int Q_CHUNK = kRowsT * 128;
  static constexpr int Q_BYTES = NCD * Q_CHUNK;
  static constexpr int KV_CHUNK = BK * 128;
  static constexpr int K_BYTES = NCD * KV_CHUNK;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + kQLoaders * Q_BYTES;
  static constexpr int OFF_V = OFF_K + K_BYTES;
  static constexpr int OFF_BAR = OFF_V + K_BYTES;
  static constexpr int SMEM = 1024 + OFF_BAR + 256;
  // TMEM: per parity p, S (and P over it) at p*256, O at p*256 + 128
  static constexpr uint32_t TMEM_COLS = 512;
};

struct Tile {
  int64_t gb;
  int g;
  int64_t b;
  int32_t first;
  int count;
};

// Walks a CTA's contiguous tile range: one binary search for the first tile,
// then (g, b) advances past empty lists as the tile index grows.
struct TileIter {
  const int32_t* __restrict__ tile_off;
  const int32_t* __restrict__ lo;
  const int32_t* __restrict__ cnt;
  int64_t n_gb, nb;
  int P;
  int64_t gb;

  __device__ __forceinline__ void seek(int32_t tile) {
    int64_t l = 0, h = n_gb;
    while (h - l > 1) {
      const int64_t m = (l + h) >> 1;
      if (tile_off[m] <= tile) l = m; else h = m;
    }
    gb = l;
  }
  // tiles must be visited in nondecreasing order
  __device__ __forceinline__ Tile at(int32_t tile) {
    while (gb + 1 < n_gb && tile_off[gb + 1] <= tile) ++gb;
    Tile r;
    r.gb = gb;
    r.g = (int)(gb / nb);
    r.b = gb % nb;
    const int32_t base = lo[gb];
    r.first = base + (tile - tile_off[gb]) * P;
    r.count = min(P, base + cnt[gb] - r.first);
    return r;
  }
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Descriptor of an MN-major operand: 64-element (128 B) rows along N, 8-row
// groups along K at 1024 B, successive 64-element N chunks `lbo` bytes apart.
__device__ __forceinline__ uint64_t umma_desc_mnmajor_sw128(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// D (TMEM) += A (TMEM, 128 lanes x 16 bf16 packed in 8 columns) * B (shared memory).
__device__ __forceinline__ void mma_bf16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

template <int D, int BK>
__global__ void __launch_bounds__(kThreadsT, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                   const uint16_t* __restrict__ q, const int32_t* __restrict__ entries,
                   const int32_t* __restrict__ lo_arr, const int32_t* __restrict__ cnt_arr,
                   const int32_t* __restrict__ tile_off, int64_t N, int H_q, int H_kv, int k, int64_t nb, int gs, int P,
                   int64_t T0, float scale_log2, uint16_t* __restrict__ part_o, float* __restrict__ part_lse,
                   DeviceStatus* st) {
  using L = AttnLayout<D, BK>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int32_t ld_t[kQLoaders][kRowsT];  // per Q loader: query position of each tile position

  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::OFF_BAR;
  auto q_full = [&](int i) { return bar0 + 8u * (0 + i); };
  auto q_empty = [&](int i) { return bar0 + 8u * (4 + i); };
  auto s_full = [&](int i) { return bar0 + 8u * (8 + i); };
  auto p_full = [&](int i) { return bar0 + 8u * (10 + i); };
  auto o_full = [&](int i) { return bar0 + 8u * (12 + i); };
  auto o_empty = [&](int i) { return bar0 + 8u * (14 + i); };
  const uint32_t kv_full = bar0 + 8u * 16;
  const uint32_t kv_empty = bar0 + 8u * 17;
  const uint32_t drain_bar = bar0 + 8u * 18;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < kQLoaders; ++i) {
      mbar_init(q_full(i), 32);
      mbar_init(q_empty(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full(i), 1);
      mbar_init(p_full(i), kSoftWarps);
      mbar_init(o_full(i), 1);
      mbar_init(o_empty(i), kSoftWarps);
    }
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    mbar_init(drain_bar, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == kWarpKv && lane == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&tmem_slot), L::TMEM_COLS);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;

  const int64_t n_gb = (int64_t)H_kv * nb;
  const int32_t total = tile_off[n_gb];
  const int32_t t_begin = (int32_t)((int64_t)total * blockIdx.x / gridDim.x);
  const int32_t t_end = (int32_t)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  const int n = t_end - t_begin;
  TileIter it{tile_off, lo_arr, cnt_arr, n_gb, nb, P, 0};
  if (n > 0) it.seek(t_begin);

  if (warp < kQLoaders) {
    // ------------------------------------------------------------ Q loader `warp`
    const int w = warp;
    int32_t* my_t = ld_t[w];
    bool ok = true;
    constexpr int CPR = D / 8;  // 16-byte chunks per Q row
    constexpr int ROWS_PER_PASS = 32 / CPR;
    const int sub_row = lane / CPR, cc = lane % CPR;
    const int ch = cc >> 3, jj = cc & 7;
    const uint32_t qdst = sbase + L::OFF_Q + w * L::Q_BYTES;
    for (int i = w; i < n && ok; i += kQLoaders) {
      const Tile tl = it.at(t_begin + i);
      const int32_t* E = entries + (int64_t)tl.g * N * k;
      for (int pp = lane; pp < P; pp += 32) my_t[pp] = pp < tl.count ? E[tl.first + pp] / k : -1;
      __syncwarp();
      int okq = 1;
      if (lane == 0) okq = mbar_wait(q_empty(w), ((i / kQLoaders) & 1) ^ 1, abort, st, 0x401) ? 1 : 0;
      if (!(ok = __shfl_sync(0xffffffffu, okq, 0) != 0)) break;
#pragma unroll 4
      for (int r0 = 0; r0 < kRowsT; r0 += ROWS_PER_PASS) {
        const int r = r0 + sub_row;
        const int pp = r / gs, hh = r % gs;
        const int32_t t = my_t[pp];
        const bool valid = t >= 0;
        const uint16_t* src = q + (((int64_t)(valid ? t : 0) * H_q + (int64_t)tl.g * gs + hh) * D + cc * 8);
        const uint32_t dst = qdst + ch * L::Q_CHUNK + r * 128 + ((jj ^ (r & 7)) << 4);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                     : "memory");
      }
      cp_async_wait_all();
      fence_proxy_async_smem();
      __syncwarp();  // my_t is rewritten for the next tile only after every lane used it
      mbar_arrive(q_full(w));
    }
    cp_async_wait_all();
  } else if (warp == kWarpKv) {
    // ------------------------------------------------------------ K/V loader
    if (lane == 0 && n > 0) {
      uint32_t runs = 0;
      int64_t prev = -1;
      int last = -1;
      bool ok = true;
      for (int i = 0; i < n && ok; ++i) {
        const Tile tl = it.at(t_begin + i);
        if (tl.gb == prev) continue;
        prev = tl.gb;
        if (!(ok = mbar_wait(kv_empty, (runs & 1) ^ 1, abort, st, 0x402))) break;
        mbar_arrive_expect_tx(kv_full, (uint32_t)(2 * L::K_BYTES));
        for (int c = 0; c < L::NCD; ++c) {
          tma_load_3d(sbase + L::OFF_K + c * L::KV_CHUNK, &tmap_k, c * 64, tl.g, (int32_t)(tl.b * BK), kv_full);
          tma_load_3d(sbase + L::OFF_V + c * L::KV_CHUNK, &tmap_v, c * 64, tl.g, (int32_t)(tl.b * BK), kv_full);
        }
        last = runs & 1;
        ++runs;
      }
      if (!ok && last >= 0) mbar_wait(kv_full, (uint32_t)last, nullptr, st, 0x4F1);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n > 0) {
      constexpr uint32_t IDESC_S = idesc_bf16_f32(kRowsT, BK);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(kRowsT, D) | (1u << 16);  // B (V) is MN-major
      uint32_t kv_cnt = 0;
      bool ok = true;
      int64_t gb_staged = -1;
      auto issue_S = [&](int j, int64_t gb_j) -> bool {
        const int qb = j % kQLoaders;
        if (!mbar_wait(q_full(qb), (j / kQLoaders) & 1, abort, st, 0x501)) return false;
        if (gb_j != gb_staged) {
          if (!mbar_wait(kv_full, kv_cnt & 1, abort, st, 0x502)) return false;
          ++kv_cnt;
          gb_staged = gb_j;
        }
        tc_fence_after();
        // S(j) reuses the columns of S/P(j-2), whose P V was issued earlier (MMAs run in issue order)
        const uint32_t d = tmem + (uint32_t)((j & 1) * 256);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int c = ks >> 2, kk = ks & 3;
          const uint64_t ad = umma_desc_kmajor(sbase + L::OFF_Q + qb * L::Q_BYTES + c * L::Q_CHUNK + kk * 32, 128);
          const uint64_t bd = umma_desc_kmajor(sbase + L::OFF_K + c * L::KV_CHUNK + kk * 32, 128);
          mma_bf16_ss(d, ad, bd, IDESC_S, ks > 0);
        }
        umma_commit(s_full(j & 1));
        umma_commit(q_empty(qb));
        return true;
      };
      auto issue_PV = [&](int i, bool last_of_block) -> bool {
        const int pb = i & 1;
        if (!mbar_wait(p_full(pb), (i >> 1) & 1, abort, st, 0x503)) return false;
        if (!mbar_wait(o_empty(pb), ((i >> 1) & 1) ^ 1, abort, st, 0x504)) return false;
        tc_fence_after();
        const uint32_t pcol = tmem + (uint32_t)(pb * 256);
        const uint32_t d = pcol + 128;
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks) {
          const uint64_t bd = umma_desc_mnmajor_sw128(sbase + L::OFF_V + ks * 16 * 128, L::KV_CHUNK);
          mma_bf16_ts(d, pcol + 8 * ks, bd, IDESC_PV, ks > 0);
        }
        umma_commit(o_full(pb));
        if (last_of_block) umma_commit(kv_empty);
        return true;
      };
      int64_t gb_cur = it.at(t_begin).gb;
      ok = issue_S(0, gb_cur);
      for (int i = 0; i < n && ok; ++i) {
        const bool has_next = i + 1 < n;
        const int64_t gb_next = has_next ? it.at(t_begin + i + 1).gb : -1;
        const bool same = has_next && gb_next == gb_cur;
        if (same && !(ok = issue_S(i + 1, gb_next))) break;
        if (!(ok = issue_PV(i, !same))) break;
        if (has_next && !same && !(ok = issue_S(i + 1, gb_next))) break;
        gb_cur = gb_next;
      }
      if (!ok) {
        umma_commit(drain_bar);
        mbar_wait(drain_bar, 0, nullptr, st, 0x5F1);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroup `par`
    const int par = (warp - kWarpSoft0) / kSoftWarps;  // tiles of this parity
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t scol = tmem + lane_base + (uint32_t)(par * 256);
    const uint32_t ocol = scol + 128;
    const int pos = row / gs, hh = row % gs;
    bool ok = true;
    for (int j = par; j < n && ok; j += 2) {
      const Tile tl = it.at(t_begin + j);
      int64_t t = -1;
      int slot = 0;
      if (pos < tl.count) {
        const int32_t e = entries[(int64_t)tl.g * N * k + tl.first + pos];
        t = e / k;
        slot = e % k;
      }
      const uint32_t ph = (j >> 1) & 1;
      if (!(ok = mbar_wait(s_full(par), ph, abort, st, 0x601))) break;
      tc_fence_after();
      // ---- softmax: max pass, then exp pass writing bf16 P over the S columns already read.
      // Columns move in pairs of 32 per TMEM wait; rows that see the whole block skip the mask.
      const int64_t key0 = tl.b * BK;
      const int lim = (int)max((int64_t)-1, min((int64_t)BK - 1, t - key0));  // last visible column
      const bool full = lim == BK - 1;
      float m = __int_as_float(0xff800000);
#pragma unroll
      for (int c = 0; c < BK / 32; c += 2) {
        uint32_t x[32], y[32];
        tmem_ld_x32(scol + c * 32, x);
        tmem_ld_x32(scol + c * 32 + 32, y);
        tmem_ld_wait();
        if (full) {
#pragma unroll
          for (int e2 = 0; e2 < 32; e2 += 2) {
            m = max3(m, __uint_as_float(x[e2]), __uint_as_float(x[e2 + 1]));
            m = max3(m, __uint_as_float(y[e2]), __uint_as_float(y[e2 + 1]));
          }
        } else {
#pragma unroll
          for (int e2 = 0; e2 < 32; ++e2) {
            if (c * 32 + e2 <= lim) m = fmaxf(m, __uint_as_float(x[e2]));
            if (c * 32 + 32 + e2 <= lim) m = fmaxf(m, __uint_as_float(y[e2]));
          }
        }
      }
      const bool empty = m == __int_as_float(0xff800000);
      const float ms = empty ? 0.f : m * scale_log2;
      float l = 0.f;
#pragma unroll
      for (int c = 0; c < BK / 32; c += 2) {
        uint32_t x[32], y[32];
        tmem_ld_x32(scol + c * 32, x);
        tmem_ld_x32(scol + c * 32 + 32, y);
        tmem_ld_wait();
        uint32_t px[16], py[16];
#pragma unroll
        for (int e2 = 0; e2 < 32; e2 += 2) {
          float a0 = ex2_approx(fmaf(__uint_as_float(x[e2]), scale_log2, -ms));
          float a1 = ex2_approx(fmaf(__uint_as_float(x[e2 + 1]), scale_log2, -ms));
          float b0 = ex2_approx(fmaf(__uint_as_float(y[e2]), scale_log2, -ms));
          float b1 = ex2_approx(fmaf(__uint_as_float(y[e2 + 1]), scale_log2, -ms));
          if (!full) {
            a0 = (c * 32 + e2 <= lim) ? a0 : 0.f;
            a1 = (c * 32 + e2 + 1 <= lim) ? a1 : 0.f;
            b0 = (c * 32 + 32 + e2 <= lim) ? b0 : 0.f;
            b1 = (c * 32 + 33 + e2 <= lim) ? b1 : 0.f;
          }
          l += (a0 + a1) + (b0 + b1);
          px[e2 >> 1] = pack_bf16x2(a0, a1);
          py[e2 >> 1] = pack_bf16x2(b0, b1);
        }
        tmem_st_x16(scol + c * 16, px);  // keys 32c..32c+31 -> packed columns 16c..16c+15
        tmem_st_x16(scol + c * 16 + 16, py);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(par));
      // ---- epilogue: normalised partial O and partial lse
      if (!(ok = mbar_wait(o_full(par), ph, abort, st, 0x602))) break;
      tc_fence_after();
      const float inv = (!empty && l > 0.f) ? 1.f / l : 0.f;
      const int64_t prow = t >= 0 ? ((t - T0) * k + slot) * H_q + (int64_t)tl.g * gs + hh : 0;
      uint16_t* dst = part_o + prow * D;
#pragma unroll
      for (int c = 0; c < D / 32; c += 2) {
        uint32_t x[2][32];
        tmem_ld_x32(ocol + c * 32, x[0]);
        tmem_ld_x32(ocol + c * 32 + 32, x[1]);
        tmem_ld_wait();
        if (t >= 0) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const uint32_t* z = x[h2] + 8 * q4;
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(z[0]) * inv, __uint_as_float(z[1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(z[2]) * inv, __uint_as_float(z[3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(z[4]) * inv, __uint_as_float(z[5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(z[6]) * inv, __uint_as_float(z[7]) * inv);
              *reinterpret_cast<uint4*>(dst + (c + h2) * 32 + q4 * 8) = v;
            }
        }
      }
      if (t >= 0)
        part_lse[prow] = (!empty && l > 0.f) ? (ms + log2f(l)) * 0.69314718055994530942f : __int_as_float(0xff800000);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty(par));
    }
  }

  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int D, int BK>
cudaError_t launch_t(const void* q, const void* kk, const void* vv, const int32_t* entries, const int32_t* lo,
                     const int32_t* cnt, const int32_t* tile_off, int64_t N, int H_q, int H_kv, int k, int64_t nb,
                     int gs, int P, int64_t T0, float scale, uint16_t* part_o, float* part_lse, DeviceStatus* st,
                     cudaStream_t s) {
  using L = AttnLayout<D, BK>;
  alignas(64) unsigned char tk[128], tv[128];
  if (!encode_tmap_3d(tk, kk, (uint64_t)D, (uint64_t)H_kv, (uint64_t)N, (uint64_t)D * 2, (uint64_t)H_kv * D * 2, 64,
                      1, BK, 128) ||
      !encode_tmap_3d(tv, vv, (uint64_t)D, (uint64_t)H_kv, (uint64_t)N, (uint64_t)D * 2, (uint64_t)H_kv * D * 2, 64,
                      1, BK, 128))
    return cudaErrorInvalidValue;
  auto kern = attn_tc_kernel<D, BK>;
  const int smem = L::SMEM > 120 * 1024 ? L::SMEM : 120 * 1024;  // one CTA per SM: TMEM is never contended
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<num_sms(), kThreadsT, smem, s>>>(*reinterpret_cast<const CUtensorMap*>(tk),
                                          *reinterpret_cast<const CUtensorMap*>(tv), (const uint16_t*)q, entries, lo,
                                          cnt, tile_off, N, H_q, H_kv, k, nb, gs, P, T0,
                                          scale * 1.4426950408889634f, part_o, part_lse, st);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_tiles(const void* q, const void* kk, const void* vv, const int32_t* entries, const int32_t* lo,
                              const int32_t* cnt, const int32_t* tile_off, int64_t N, int H_q, int H_kv, int d,
                              int Bk, int k, int64_t nb, int gs, int P, int64_t T0, float scale, uint16_t* part_o,
                              float* part_lse, DeviceStatus* st, cudaStream_t s) {
  if (d == 64 && Bk == 64)
    return launch_t<64, 64>(q, kk, vv, entries, lo, cnt, tile_off, N, H_q, H_kv, k, nb, gs, P, T0, scale, part_o,
                            part_lse, st, s);
  if (d == 64)
    return launch_t<64, 128>(q, kk, vv, entries, lo, cnt, tile_off, N, H_q, H_kv, k, nb, gs, P, T0, scale, part_o,
                             part_lse, st, s);
  if (Bk == 64)
    return launch_t<128, 64>(q, kk, vv, entries, lo, cnt, tile_off, N, H_q, H_kv, k, nb, gs, P, T0, scale, part_o,
                             part_lse, st, s);
  return launch_t<128, 128>(q, kk, vv, entries, lo, cnt, tile_off, N, H_q, H_kv, k, nb, gs, P, T0, scale, part_o,
                            part_lse, st, s);
}

}  // namespace msa
