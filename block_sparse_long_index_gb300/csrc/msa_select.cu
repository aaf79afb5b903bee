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

template <int DI>
struct SelectLayout {
  static constexpr int CH_E = DI >= 64 ? 64 : DI;  // elements per swizzled row chunk
  static constexpr int CH_B = CH_E * 2;             // 128 or 64 bytes
  static constexpr int NCH = DI / CH_E;
  static constexpr int A_CHUNK = kRows * CH_B;
  static constexpr int B_CHUNK = kKeys * CH_B;
  static constexpr int A_BYTES = kMaxGpc * NCH * A_CHUNK;
  static constexpr int STAGE_BYTES = NCH * B_CHUNK;
  static constexpr int STAGES_FIT = (200 * 1024 - A_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 4 ? 4 : STAGES_FIT;  // k^I ring depth
  static constexpr int KSTEPS = CH_E / 16;
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

template <int DI, int CAP>
__global__ void __launch_bounds__(kThreads, 1)
    select_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     int64_t N, int G, int gpc, int Bk, int k, int32_t* __restrict__ block_idx, DeviceStatus* st) {
  using L = SelectLayout<DI>;
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
        const int64_t nkt = key_tiles(qb, Bk);
        if (nkt == 0) continue;
        if (!(ok = mbar_wait(a_empty, (a_glob & 1) ^ 1, abort, st, 0x101))) break;
        mbar_arrive_expect_tx(a_full, (uint32_t)(gpc * L::NCH * L::A_CHUNK));
        for (int gi = 0; gi < gpc; ++gi)
          for (int c = 0; c < L::NCH; ++c)
            tma_load_2d(smem_u32(sA + (gi * L::NCH + c) * L::A_CHUNK), &tmap_q,
                        (gq * gpc + gi) * DI + c * L::CH_E, (int32_t)(qb * kRows), a_full);
        a_last = a_glob & 1;
        ++a_glob;
        for (int64_t kt = 0; kt < nkt; ++kt, ++kt_glob) {
          const int s = kt_glob % kStages;
          const uint32_t ph = (kt_glob / kStages) & 1;
          if (!(ok = mbar_wait(empty_bar(s), ph ^ 1, abort, st, 0x102))) break;
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
      constexpr uint32_t IDESC = idesc_bf16_f32(kRows, kKeys);
      uint32_t kt_glob = 0, a_glob = 0;
      uint32_t uses0 = 0, uses1 = 0;  // fills of accumulator buffers 0 and 1 so far
      int64_t r = 0, j;
      bool ok = true;
      while (ok && next_item(r, n_items, j)) {
        const int64_t qb = n_qt - 1 - j / n_gq;
        const int64_t nkt = key_tiles(qb, Bk);
        if (nkt == 0) continue;
        if (!(ok = mbar_wait(a_full, a_glob & 1, abort, st, 0x201))) break;
        tc_fence_after();
        for (int64_t kt = 0; kt < nkt; ++kt, ++kt_glob) {
          const int s = kt_glob % kStages;
          if (!(ok = mbar_wait(full_bar(s), (kt_glob / kStages) & 1, abort, st, 0x202))) break;
          for (int gi = 0; gi < gpc && ok; ++gi) {
            const int buf = gpc == 2 ? gi : (int)(kt_glob & 1);
            const uint32_t use = buf ? uses1 : uses0;
            if (!(ok = mbar_wait(acc_empty(buf), (use & 1) ^ 1, abort, st, 0x203))) break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(buf * kKeys);
#pragma unroll
            for (int c = 0; c < L::NCH; ++c)
#pragma unroll
              for (int kk = 0; kk < L::KSTEPS; ++kk) {
                const uint64_t ad = umma_desc_kmajor(smem_u32(sA + (gi * L::NCH + c) * L::A_CHUNK + kk * 32), L::CH_B);
                const uint64_t bd =
                    umma_desc_kmajor(smem_u32(sB + s * L::STAGE_BYTES + c * L::B_CHUNK + kk * 32), L::CH_B);
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
      const int64_t nkt = key_tiles(qb, Bk);
      const int64_t t = qb * kRows + row;
      const int64_t local = t / Bk;
      top.init(k - 1);
      for (int64_t kt = 0; kt < nkt; ++kt, ++kt_glob) {
        const int buf = gpc == 2 ? gi : (int)(kt_glob & 1);
        const uint32_t use = buf ? uses1 : uses0;
        if (!(ok = mbar_wait(acc_full(buf), use & 1, abort, st, 0x301))) break;
        if (buf) ++uses1; else ++uses0;
        tc_fence_after();
        // the tile's four 64-key quarters in turn; a block's maximum is offered
        // as soon as its quarters are done (Bk = 128: two, Bk = 64: one)
        const uint32_t col = tmem + lane_base + (uint32_t)(buf * kKeys);
        float mb = __int_as_float(0xff800000);
#pragma unroll 1
        for (int h = 0; h < 4; ++h) {
          uint32_t x[32], y[32];
          tmem_ld_x32(col + 64 * h, x);
          tmem_ld_x32(col + 64 * h + 32, y);
          tmem_ld_wait();
          if (h == 3) {  // the whole tile is in registers or reduced: release TMEM
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(buf));
          }
#pragma unroll
          for (int i = 0; i < 32; i += 2) mb = max3(mb, __uint_as_float(x[i]), __uint_as_float(x[i + 1]));
#pragma unroll
          for (int i = 0; i < 32; i += 2) mb = max3(mb, __uint_as_float(y[i]), __uint_as_float(y[i + 1]));
          if (Bk == 64 || (h & 1)) {
            const int b = Bk == 128 ? (int)(2 * kt) + (h >> 1) : (int)(4 * kt) + h;
            if (b < local) top.insert(mb, b);
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

template <int DI, int CAP>
cudaError_t launch_t(const void* q_idx, const void* k_idx, int64_t N, int G, int gpc, int Bk, int k,
                     int32_t* block_idx, DeviceStatus* st, cudaStream_t s) {
  using L = SelectLayout<DI>;
  CUtensorMap tq, tk;
  if (!encode_tmap_2d(&tq, q_idx, (uint64_t)G * DI, (uint64_t)N, (uint64_t)G * DI * 2, L::CH_E, kRows, L::CH_B))
    return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tk, k_idx, (uint64_t)DI, (uint64_t)N, (uint64_t)DI * 2, L::CH_E, kKeys, L::CH_B))
    return cudaErrorInvalidValue;
  auto kern = select_tc_kernel<DI, CAP>;
  // more than half of an SM's shared memory: one CTA per SM, so the 512 TMEM columns are always free
  const int smem = L::SMEM > 120 * 1024 ? L::SMEM : 120 * 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t n_items = ((N + kRows - 1) / kRows) * (G / gpc);
  const int grid = (int)(n_items < num_sms() ? n_items : num_sms());
  kern<<<grid, kThreads, smem, s>>>(tq, tk, N, G, gpc, Bk, k, block_idx, st);
  return cudaGetLastError();
}

template <int DI>
cudaError_t launch_cap(const void* q_idx, const void* k_idx, int64_t N, int G, int gpc, int Bk, int k,
                       int32_t* block_idx, DeviceStatus* st, cudaStream_t s) {
  const int km1 = k - 1;
  if (km1 <= 4) return launch_t<DI, 4>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, st, s);
  if (km1 <= 8) return launch_t<DI, 8>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, st, s);
  if (km1 <= 16) return launch_t<DI, 16>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, st, s);
  return launch_t<DI, 32>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, st, s);
}

}  // namespace

cudaError_t launch_select(const void* q_idx, const void* k_idx, int64_t N, int G, int d_I, int Bk, int k,
                          int32_t* block_idx, DeviceStatus* st, cudaStream_t s) {
  const int gpc = (G % 2 == 0) ? 2 : 1;
  if (d_I == 32) return launch_cap<32>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, st, s);
  if (d_I == 64) return launch_cap<64>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, st, s);
  return launch_cap<128>(q_idx, k_idx, N, G, gpc, Bk, k, block_idx, st, s);
}

}  // namespace msa
