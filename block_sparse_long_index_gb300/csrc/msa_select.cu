// msa_select_blocks: index scoring + block max-pooling + local-pinned top-k
// on the 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA).
//
// "MSA" study note 2-3 (s = q^I.k^I / sqrt(d_I); S = max over the block's
// tokens j <= t; set = local block + top-k), 3-2 (max-pooling), 3-5
// (exp-free top-k on raw scores) and Flash-MSA "プロキシアテンション"
// (per-tile maxima inserted into a register top-k while sweeping key tiles;
// local block pinned).
//
// Work item = (query tile of 128 rows, pair of GQA groups).  The index key
// is shared by all groups, so one 256-key tile of k^I staged in shared memory
// feeds GPC (<= 2) MMAs of 128 x 256 x d_I, one per group (256-wide B tiles
// run the tensor core closer to its peak than 128-wide ones):
//   warp 0      TMA producer: the item's q^I tiles (A, resident for the
//               item) and a ring of k^I tiles (B, 2 to 4 stages), swizzled;
//   warp 1      allocates TMEM; lane 0 issues tcgen05.mma into one 256-column
//               fp32 accumulator per group (with one group, two buffers
//               alternate), so one group's MMAs run while the other's scores
//               are reduced, and commits completion to mbarriers;
//   warps 2..9  epilogue: each thread owns one query row (a TMEM lane) of one
//               group, loads its 256 scores with tcgen05.ld, reduces them with
//               3-input max into block maxima (one per Bk-block of the tile)
//               and offers (max, block) to its register top-(k-1) list.
//               Scores never leave the SM.
// The same kernel runs on FP8 E4M3 index inputs (chipsbuilder "Co-Design Del
// Kernel": FP8 among the kernel's precisions): tcgen05.mma kind::f8f6f4 takes
// 32 bytes of K per instruction as kind::f16 does, so the shared-memory tiles,
// descriptors and K steps are the same in bytes and a tile of d_I = 128 is one
// 128-byte swizzle atom per row; the tensor core runs twice the multiply-adds
// per instruction.
// Only blocks b < local(t) are candidates: every token of such a block is
// visible (j <= t), so no causal mask is applied; the local block is written
// directly as slot 0.  Items are visited longest-first in a snake order over
// the persistent CTAs so the causal triangle balances.  Every wait is bounded
// (about 2 s); on expiry the kernel raises the timeout flag, drains its own
// asynchronous work and exits.
#include "msa_sm100.cuh"

namespace msa {

namespace {

using namespace sm100;

constexpr int kRows = 128;     // query rows per tile = MMA M
constexpr int kKeys = 256;     // keys per tile = MMA N
constexpr int kMaxGpc = 2;     // groups per work item
constexpr int kEpiWarps = 4 * kMaxGpc;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr uint32_t kHint = 20000;  // ns: waiting warps sleep in try_wait instead of spinning

template <int DI, bool F8>
struct SelectLayout {
  static constexpr int ESZ = F8 ? 1 : 2;              // bytes per element
  static constexpr int RB = DI * ESZ;                 // bytes per row
  static constexpr int CH_B = RB >= 128 ? 128 : RB;   // bytes per swizzled row chunk
  static constexpr int CH_E = CH_B / ESZ;             // elements per chunk
  static constexpr int NCH = RB / CH_B;
  static_assert(CH_B == 64 || CH_B == 128, "rows of 64 or 128 bytes per swizzle atom");
  static constexpr int A_CHUNK = kRows * CH_B;
  static constexpr int B_CHUNK = kKeys * CH_B;
  static constexpr int A_BYTES = kMaxGpc * NCH * A_CHUNK;
  static constexpr int STAGE_BYTES = NCH * B_CHUNK;
  static constexpr int STAGES_FIT = (200 * 1024 - A_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 4 ? 4 : STAGES_FIT;  // k^I ring depth
  static constexpr int KSTEPS = CH_B / 32;  // 32 bytes of K per MMA
  static constexpr int BAR_BYTES = 256;
  static constexpr int SMEM = 1024 + A_BYTES + STAGES * STAGE_BYTES + BAR_BYTES;
  static_assert(STAGES >= 2, "k^I ring needs two stages");
};

__device__ __forceinline__ bool next_item(int64_t& r, int64_t n_items, int64_t& j) {
  // snake order over the persistent CTAs: round r visits items [r*grid, (r+1)*grid)
  while (true) {
    const int64_t base = r * gridDim.x;
    if (base >= n_items) return false;
    const int64_t c = (r & 1) ? (int64_t)gridDim.x - 1 - blockIdx.x : (int64_t)blockIdx.x;
    ++r;
    j = base + c;
    if (j < n_items) return true;
  }
}

// Key tiles a query tile needs: the 256-key tiles holding blocks before the
// last row's local block (for Bk = 64 the second half of the query tile also
// takes block 2qb).  Keys past that (a local block, or past N: zero fill) are
// scored but never offered.
__device__ __forceinline__ int64_t key_tiles(int64_t qb, int Bk) {
  const int64_t key_limit = qb * kRows + (Bk == 128 ? 0 : 64);
  return (key_limit + kKeys - 1) / kKeys;
}

// First key tile a query tile needs when several sequences share the cells
// (blk_lo[b] = first block of block b's sequence): the tile holding the first
// block of its first row's sequence; 0 for one sequence.
__device__ __forceinline__ int64_t first_key_tile(const int32_t* blk_lo, int64_t qb, int Bk) {
  return blk_lo ? (int64_t)__ldg(blk_lo + qb * kRows / Bk) * Bk / kKeys : 0;
}

template <int DI, int CAP, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    select_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     int64_t N, int G, int gpc, int Bk, int k, int32_t* __restrict__ block_idx,
                     const int32_t* __restrict__ blk_lo, DeviceStatus* st) {
  using L = SelectLayout<DI, F8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + L::A_BYTES;
  constexpr int kStages = L::STAGES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + kStages * L::STAGE_BYTES);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  const uint32_t a_full = bar0 + 8u * (2 * kStages);
  const uint32_t a_empty = a_full + 8u;
  auto acc_full = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (2 * kStages + 4 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 6);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr uint32_t tmem_cols = 2 * kKeys;  // accumulator buffer b at columns kKeys * b

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(a_full, 1);
    mbar_init(a_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 4);  // the four warps of the group that drains it
    }
    mbar_init(drain_bar, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), tmem_cols);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;

  const int64_t n_qt = (N + kRows - 1) / kRows;
  const int n_gq = G / gpc;
  const int64_t n_items = n_qt * n_gq;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t kt_glob = 0, a_glob = 0;
      int last_phase[kStages];
      for (int s = 0; s < kStages; ++s) last_phase[s] = -1;
      int a_last = -1;
      int64_t r = 0, j;
      bool ok = true;
      while (ok && next_item(r, n_items, j)) {
        const int64_t qb = n_qt - 1 - j / n_gq;
        const int gq = (int)(j % n_gq);
        const int64_t nkt = key_tiles(qb, Bk), kt0 = first_key_tile(blk_lo, qb, Bk);
        if (nkt <= kt0) continue;
        if (!(ok = mbar_wait(a_empty, (a_glob & 1) ^ 1, abort, st, 0x101, kHint))) break;
        mbar_arrive_expect_tx(a_full, (uint32_t)(gpc * L::NCH * L::A_CHUNK));
        for (int gi = 0; gi < gpc; ++gi)
          for (int c = 0; c < L::NCH; ++c)
            tma_load_2d(smem_u32(sA + (gi * L::NCH + c) * L::A_CHUNK), &tmap_q,
                        (gq * gpc + gi) * DI + c * L::CH_E, (int32_t)(qb * kRows), a_full);
        a_last = a_glob & 1;
        ++a_glob;
        for (int64_t kt = kt0; kt < nkt; ++kt, ++kt_glob) {
          const int s = kt_glob % kStages;
          const uint32_t ph = (kt_glob / kStages) & 1;
          if (!(ok = mbar_wait(empty_bar(s), ph ^ 1, abort, st, 0x102, kHint))) break;
          mbar_arrive_expect_tx(full_bar(s), (uint32_t)L::STAGE_BYTES);
          for (int c = 0; c < L::NCH; ++c)
            tma_load_2d(smem_u32(sB + s * L::STAGE_BYTES + c * L::B_CHUNK), &tmap_k, c * L::CH_E,
                        (int32_t)(kt * kKeys), full_bar(s));
          last_phase[s] = (int)ph;
        }
      }
      if (!ok) {  // let our own copies land before the CTA exits
        for (int s = 0; s < kStages; ++s)
          if (last_phase[s] >= 0) mbar_wait(full_bar(s), (uint32_t)last_phase[s], nullptr, st, 0x1F1);
        if (a_last >= 0) mbar_wait(a_full, (uint32_t)a_last, nullptr, st, 0x1F2);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = F8 ? idesc_e4m3_f32(kRows, kKeys) : idesc_bf16_f32(kRows, kKeys);
      uint32_t kt_glob = 0, a_glob = 0;
      uint32_t uses0 = 0, uses1 = 0;  // fills of accumulator buffers 0 and 1 so far
      int64_t r = 0, j;
      bool ok = true;
      while (ok && next_item(r, n_items, j)) {
        const int64_t qb = n_qt - 1 - j / n_gq;
        const int64_t nkt = key_tiles(qb, Bk), kt0 = first_key_tile(blk_lo, qb, Bk);
        if (nkt <= kt0) continue;
        if (!(ok = mbar_wait(a_full, a_glob & 1, abort, st, 0x201, kHint))) break;
        tc_fence_after();
        for (int64_t kt = kt0; kt < nkt; ++kt, ++kt_glob) {
          const int s = kt_glob % kStages;
          if (!(ok = mbar_wait(full_bar(s), (kt_glob / kStages) & 1, abort, st, 0x202, kHint))) break;
          for (int gi = 0; gi < gpc && ok; ++gi) {
            const int buf = gpc == 2 ? gi : (int)(kt_glob & 1);
            const uint32_t use = buf ? uses1 : uses0;
            if (!(ok = mbar_wait(acc_empty(buf), (use & 1) ^ 1, abort, st, 0x203, kHint))) break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(buf * kKeys);
#pragma unroll
            for (int c = 0; c < L::NCH; ++c)
#pragma unroll
              for (int kk = 0; kk < L::KSTEPS; ++kk) {
                const uint64_t ad = umma_desc_kmajor(smem_u32(sA + (gi * L::NCH + c) * L::A_CHUNK + kk * 32), L::CH_B);
                const uint64_t bd =
                    umma_desc_kmajor(smem_u32(sB + s * L::STAGE_BYTES + c * L::B_CHUNK + kk * 32), L::CH_B);
                if constexpr (F8)
                  mma_e4m3_ss(d, ad, bd, IDESC, (c | kk) != 0);
                else
                  mma_bf16_ss(d, ad, bd, IDESC, (c | kk) != 0);
              }
            umma_commit(acc_full(buf));
            if (buf) ++uses1; else ++uses0;
          }
          if (!ok) break;
          umma_commit(empty_bar(s));
        }
        if (!ok) break;
        umma_commit(a_empty);
        ++a_glob;
      }
      if (!ok) {  // wait for the MMAs already issued before TMEM is released
        umma_commit(drain_bar);
        mbar_wait(drain_bar, 0, nullptr, st, 0x2F1);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
    const int gi = (warp - 2) >> 2;        // the group (of the item's pair) this warp reduces
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    uint32_t kt_glob = 0;
    uint32_t uses0 = 0, uses1 = 0;
    int64_t r = 0, j;
    bool ok = gi < gpc;  // with one group per item, the second group's warps have nothing to do
    TopK<CAP> top;
    while (ok && next_item(r, n_items, j)) {
      const int64_t qb = n_qt - 1 - j / n_gq;
      const int gq = (int)(j % n_gq);
      const int64_t nkt = key_tiles(qb, Bk), kt0 = first_key_tile(blk_lo, qb, Bk);
      const int64_t t = qb * kRows + row;
      const int64_t local = t / Bk;
      // candidates: blocks [lo, local) of the row's own sequence
      const int64_t lo = (blk_lo && t < N) ? (int64_t)__ldg(blk_lo + local) : 0;
      top.init(k - 1);
      for (int64_t kt = kt0; kt < nkt; ++kt, ++kt_glob) {
        const int buf = gpc == 2 ? gi : (int)(kt_glob & 1);
        const uint32_t use = buf ? uses1 : uses0;
        if (!(ok = mbar_wait(acc_full(buf), use & 1, abort, st, 0x301, kHint))) break;
        if (buf) ++uses1; else ++uses0;
        tc_fence_after();
        // the tile's four 64-key quarters in turn, the next quarter's TMEM
        // loads in flight while this one is reduced; a block's maximum is
        // offered as soon as its quarters are done (Bk = 128: two, Bk = 64:
        // one).  Four independent max chains keep the reduction short.
        const uint32_t col = tmem + lane_base + (uint32_t)(buf * kKeys);
        float mb = __int_as_float(0xff800000);
        uint32_t xq[2][2][32];
        tmem_ld_x32(col, xq[0][0]);
        tmem_ld_x32(col + 32, xq[0][1]);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t (&x)[32] = xq[h & 1][0];
          uint32_t (&y)[32] = xq[h & 1][1];
          tmem_ld_wait();
          reg_fence32(x);
          reg_fence32(y);
          if (h == 3) {  // the whole tile is in registers or reduced: release TMEM
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(buf));
          } else {
            tmem_ld_x32(col + 64 * (h + 1), xq[(h + 1) & 1][0]);
            tmem_ld_x32(col + 64 * (h + 1) + 32, xq[(h + 1) & 1][1]);
          }
          float m4[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) m4[c] = max3(__uint_as_float(x[2 * c]), __uint_as_float(x[2 * c + 1]), mb);
#pragma unroll
          for (int i = 8; i < 32; i += 8)
#pragma unroll
            for (int c = 0; c < 4; ++c)
              m4[c] = max3(m4[c], __uint_as_float(x[i + 2 * c]), __uint_as_float(x[i + 2 * c + 1]));
#pragma unroll
          for (int i = 0; i < 32; i += 8)
#pragma unroll
            for (int c = 0; c < 4; ++c)
              m4[c] = max3(m4[c], __uint_as_float(y[i + 2 * c]), __uint_as_float(y[i + 2 * c + 1]));
          mb = max3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
          if (Bk == 64 || (h & 1)) {
            const int b = Bk == 128 ? (int)(2 * kt) + (h >> 1) : (int)(4 * kt) + h;
            if (b < local && b >= lo) top.insert(mb, b);
            mb = __int_as_float(0xff800000);
          }
        }
      }
      if (!ok) break;
      if (t < N) {
        int32_t* out = block_idx + ((int64_t)(gq * gpc + gi) * N + t) * k;
        out[0] = (int32_t)local;
        if (k > 1) top.emit(k - 1, out + 1);
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

template <int DI, int CAP, bool F8>
cudaError_t launch_t(const void* q_idx, const void* k_idx, int64_t N, int G, int gpc, int Bk, int k,
                     int32_t* block_idx, const int32_t* blk_lo, DeviceStatus* st, cudaStream_t s) {
  using L = SelectLayout<DI, F8>;
  CUtensorMap tq, tk;
  if (!encode_tmap_2d(&tq, q_idx, (uint64_t)G * DI, (uint64_t)N, (uint64_t)G * L::RB, L::CH_E, kRows, L::CH_B,
                      L::ESZ))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tk, k_idx, (uint64_t)DI, (uint64_t)N, (uint64_t)L::RB, L::CH_E, kKeys, L::CH_B, L::ESZ))
    return cudaErrorInvalidValue;
  auto kern = select_tc_kernel<DI, CAP, F8>;
  // more than half of an SM's shared memory: one CTA per SM, so the 512 TMEM columns are always free
  const int smem = L::SMEM > 120 * 1024 ? L::SMEM : 120 * 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t n_items = ((N + kRows - 1) / kRows) * (G / gpc);
  const int grid = (int)(n_items < num_sms() ? n_items : num_sms());
  kern<<<grid, kThreads, smem, s>>>(tq, tk, N, G, gpc, Bk, k, block_idx, blk_lo, st);
  return cudaGetLastError();
}

template <int DI, bool F8>
cudaError_t launch_cap(const void* q_idx, const void* k_idx, int64_t N, int G, int gpc, int Bk, int k,
                       int32_t* block_idx, const int32_t* blk_lo, DeviceStatus* st, cudaStream_t s) {
  const int km1 = k - 1;
  if (km1 <= 4) return launch_t<DI, 4, F8>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, blk_lo, st, s);
  if (km1 <= 8) return launch_t<DI, 8, F8>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, blk_lo, st, s);
  if (km1 <= 16) return launch_t<DI, 16, F8>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, blk_lo, st, s);
  return launch_t<DI, 32, F8>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, blk_lo, st, s);
}

// blk_lo[b] = first block of the sequence whose cells hold block b.  Sequence
// s holds cells [cu[s], cu[s+1]); every cu[s] must be a multiple of Bk with
// cu[0] = 0, non-decreasing, cu[S] <= N.  Blocks past cu[S] belong to no
// sequence (blk_lo[b] = b: the local block only).  A cu that breaks those
// rules sets the device error word; every block then keeps only its local
// block.
__global__ void varlen_blocks_kernel(const int32_t* __restrict__ cu, int S, int64_t N, int Bk, int64_t nb,
                                     int32_t* __restrict__ blk_lo, DeviceStatus* st) {
  __shared__ int bad;
  if (threadIdx.x == 0) {
    int b_ = cu[0] != 0;
    for (int i = 0; i < S && !b_; ++i) b_ = cu[i + 1] < cu[i] || (cu[i + 1] % Bk) != 0;
    b_ = b_ || (int64_t)cu[S] > N;
    bad = b_;
    if (b_ && blockIdx.x == 0) raise_error(st, kErrBadIndex, 4u);
  }
  __syncthreads();
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < nb; b += (int64_t)gridDim.x * blockDim.x) {
    int32_t lo = (int32_t)b;
    if (!bad && b * Bk < (int64_t)cu[S]) {
      int a = 0, z = S;  // the last s with cu[s] <= b * Bk (cu[0] = 0 <= b * Bk)
      while (z - a > 1) {
        const int m = (a + z) >> 1;
        if ((int64_t)cu[m] <= b * Bk) a = m; else z = m;
      }
      lo = cu[a] / Bk;
    }
    blk_lo[b] = lo;
  }
}

// y = E4M3 code of (bf16 x) * scale, nearest with ties to even, saturated at
// +-448 (cvt.rn.satfinite); eight elements (16 bytes in, 8 out) per step when
// both pointers allow it.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(256) quantize_e4m3_kernel(const uint16_t* __restrict__ x, int64_t n, float scale,
                                                            uint8_t* __restrict__ y, int vec) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t done = 0;
  if (vec) {
    const int64_t n8 = n / 8;
    for (int64_t i = i0; i < n8; i += stride) {
      const uint4 v = ldg_stream_16(x + 8 * i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t p[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) p[j] = cvt_e4m3x2(__fmul_rn(bf16_hi(w[j]), scale), __fmul_rn(bf16_lo(w[j]), scale));
      *reinterpret_cast<uint2*>(y + 8 * i) = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
    }
    done = n8 * 8;
  }
  for (int64_t i = done + i0; i < n; i += stride)
    y[i] = (uint8_t)(cvt_e4m3x2(0.f, __fmul_rn(__uint_as_float((uint32_t)x[i] << 16), scale)) & 0xFFu);
}

}  // namespace

cudaError_t launch_select(const void* q_idx, const void* k_idx, int64_t N, int G, int d_I, int Bk, int k,
                          int32_t* block_idx, DeviceStatus* st, cudaStream_t s, bool f8, const int32_t* blk_lo) {
  const int gpc = (G % 2 == 0) ? 2 : 1;
  if (f8) {  // d_I of 64 or 128 (64- or 128-byte rows)
    if (d_I == 64) return launch_cap<64, true>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, blk_lo, st, s);
    if (d_I == 128) return launch_cap<128, true>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, blk_lo, st, s);
    return cudaErrorInvalidValue;
  }
  if (d_I == 32) return launch_cap<32, false>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, blk_lo, st, s);
  if (d_I == 64) return launch_cap<64, false>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, blk_lo, st, s);
  return launch_cap<128, false>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, blk_lo, st, s);
}

cudaError_t launch_varlen_blocks(const int32_t* cu_seqlens, int S, int64_t N, int Bk, int32_t* blk_lo,
                                 DeviceStatus* st, cudaStream_t s) {
  const int64_t nb = (N + Bk - 1) / Bk;
  int64_t blocks = (nb + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  varlen_blocks_kernel<<<(unsigned)blocks, 256, 0, s>>>(cu_seqlens, S, N, Bk, nb, blk_lo, st);
  return cudaGetLastError();
}

cudaError_t launch_quantize_e4m3(const void* x, int64_t n, float scale, void* y, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int vec = ((reinterpret_cast<uintptr_t>(x) & 15u) == 0 && (reinterpret_cast<uintptr_t>(y) & 7u) == 0) ? 1 : 0;
  const int64_t per_thread = vec ? 8 : 1;
  int64_t blocks = (n / per_thread + 255) / 256;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  quantize_e4m3_kernel<<<(unsigned)blocks, 256, 0, s>>>((const uint16_t*)x, n, scale, (uint8_t*)y, vec);
  return cudaGetLastError();
}

}  // namespace msa
