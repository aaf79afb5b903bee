// KV-outer attention tiles on the 5th-generation tensor cores.
//
// "MSA" study note 3-3 "Main Branch" (exact softmax over the selected
// support, per-head weights, group-shared blocks) and 3-5 (KV-outer: the
// queries that chose a KV block are concatenated into one large MMA that
// reuses the block from on-chip memory; hot blocks pre-chunked into tiles).
//
// A tile is (group g, block b, up to P = 16 ppr query positions that chose
// b), ppr = 8 / gs: its 128 MMA rows are (position pp, head hh < gs) -> row
// gs pp + hh, so every row is a real (position, head) whatever the group
// size, and one 8-row swizzle atom holds ppr positions.  Per tile:
//   S = Q K_b^T (128 x Bk fp32 in TMEM), causal mask j <= t, row max m and
//   P = 2^(s log2e / sqrt(d) - m) (bf16, each half of the keys written back
//   over the first columns of that half of S),
//   O = P V_b (128 x d fp32 in TMEM, P read from TMEM as the A operand); the
//   row's un-normalised O goes out in bf16 and its (m, l = sum P) in fp32, so
//   the combine divides once per (t, h) by the merged sum.
// Roles (512 threads):
//   warp 3        copies each tile's ppr 128-byte records (query positions,
//                 slots) from the schedule into an 8-slot shared ring;
//   warp 0        Q loader: gathers a tile's Q rows with TMA boxes per
//                 position (gs heads x 64 dims, or all 8 heads x d in one box
//                 when gs = 8) into one of three position-major,
//                 128B-swizzled K-major Q buffers;
//   warp 1        TMEM owner; lane 0 issues tcgen05.mma.  S/P and O have two
//                 TMEM buffers each, so S runs one tile ahead of P V and the
//                 epilogue drains O(i-1) while PV(i) runs: per tile i it issues
//                 S(i+1) if it uses i's K/V block, then PV(i);
//   warp 2        K/V loader: one TMA load of K_b and V_b per run of tiles of
//                 the same block, released after the run's last P V;
//   warps 4..11   two softmax warpgroups, both on every tile: each takes one
//                 half of the key columns and writes its P over that half;
//   warps 12..15  epilogue warpgroup: O -> bf16 in a position-major, swizzled
//                 shared tile, written out by one TMA store box per position
//                 (its gs heads x d).
// A position's gs rows of an atom sit at byte (pp % ppr) gs 128 of atom
// pp / ppr; TMA applies the 128-byte swizzle by shared-memory address, so a
// box of gs rows written there lands exactly where the 8-row atom has them.
// Buffer reuse needs no extra waits: S(j) is issued after PV(j-2) (tensor
// core operations run in issue order), and each barrier phase a role waits
// for cannot be overtaken by the next one (the next use of a buffer depends,
// through the issue order, on the consumer having passed it).  K_b, Q feed
// the tensor cores as K-major shared-memory operands, V_b as an MN-major one
// (d contiguous), P from TMEM.  Every wait is bounded; on expiry the kernel
// flags a timeout, drains its own async work and exits.
#include <math.h>

#include "msa_sm100.cuh"

namespace msa {

namespace {

using namespace sm100;

constexpr int kRowsT = 128;   // MMA rows per tile
constexpr int kPosT = 16;     // query positions per tile
constexpr int kQBufs = 3;     // Q buffers in shared memory
constexpr int kSBufs = 2;     // S/P buffers in TMEM (one per softmax warpgroup)
constexpr int kOBufs = 2;     // O buffers in TMEM
constexpr int kMeta = 8;      // tile metadata slots
constexpr int kWarpLoad = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpKv = 2;
constexpr int kWarpMeta = 3;
constexpr int kWarpSoft0 = 4;
constexpr int kWarpEpi0 = 12;
constexpr int kThreadsT = 16 * 32;
constexpr int kSoftWarps = 4;  // per warpgroup
constexpr int kEpiWarps = 4;
// Q loader, K/V loader, MMA issuer, the eight softmax warps, epilogue store issuer
constexpr int kMetaReaders = 1 + 1 + 1 + 2 * kSoftWarps + 1;
static_assert(kPosT == kTilePositions, "tile records hold 16 positions");

// Q and O tiles in shared memory are atom-major: 8-row group a (ppr positions)
// holds its d/64 chunks of 8 rows x 128 bytes (one 128B-swizzle atom each) in
// POS_BYTES, so rows 8a..8a+7 of K-chunk c sit at a * POS_BYTES + c * 1024.
template <int D, int BK>
struct AttnLayout {
  static constexpr int NCD = D / 64;                // 64-column chunks of d
  static constexpr int POS_BYTES = NCD * 1024;
  static constexpr int Q_BYTES = kPosT * POS_BYTES;
  static constexpr int KV_CHUNK = BK * 128;
  static constexpr int K_BYTES = NCD * KV_CHUNK;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + kQBufs * Q_BYTES;
  static constexpr int OFF_V = OFF_K + K_BYTES;
  static constexpr int OFF_STG = OFF_V + K_BYTES;   // bf16 O of one tile, same layout as Q
  static constexpr int OFF_BAR = OFF_STG + Q_BYTES;
  static constexpr int SMEM = 1024 + OFF_BAR + 512;
  // TMEM: S/P buffer j at 128 j, O buffer j at 256 + 128 j
  static constexpr uint32_t TMEM_O = 256;
  static constexpr uint32_t TMEM_COLS = 512;
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}
// Plain bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            int32_t w, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y, int32_t z,
                                             int32_t w) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];\n" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}
// The CTAs split the tile list by weight, not by count: a (group, block) run
// weighs its tiles plus kRunWeight more for its start (the K/V load and the
// run's leading diagonal tiles, whose masked softmax is slower).  Timed per
// CTA at 128K, an equal count of tiles left the CTAs that hold the short runs
// of the late blocks 1.2-1.5 ms behind the median (the per-CTA end time fits
// 4.7 us per run on top of the tiles).  A block inside the query slab
// [T0, T1) has the diagonal tiles of its own positions; a block before the
// slab (later slabs of a long prefill) has none and weighs less; a block past
// the slab has no tiles at all and weighs nothing.  With runs in (group,
// block) order, r = g nb + b, and b0 = T0 / Bk, b1 = ceil(T1 / Bk), the runs
// before r number F(r) = g b0 + min(b, b0) before the slab and
// I(r) = g (b1 - b0) + clamp(b - b0, 0, b1 - b0) inside it, so run r starts at
// weight W(r) = tile_off[r] + rf F(r) + rd I(r).  A CTA's first tile is the
// one at weight W_total c / grid, found by a 32-ary search of one warp.
struct RunWeights {
  int64_t nb, b0, b1, rd, rf;  // blocks per group, the slab's blocks [b0, b1), start weight in / before it
  __device__ __forceinline__ int64_t start(const int32_t* tile_off, int64_t r) const {
    const int64_t g = r / nb, b = r % nb;
    const int64_t before = g * b0 + min(b, b0);
    const int64_t in = g * (b1 - b0) + min(max(b - b0, (int64_t)0), b1 - b0);
    return (int64_t)tile_off[r] + rf * before + rd * in;
  }
  __device__ __forceinline__ int64_t own(int64_t r) const {
    const int64_t b = r % nb;
    return b < b0 ? rf : b < b1 ? rd : 0;
  }
};
__device__ __forceinline__ int64_t tile_at_weight(const int32_t* __restrict__ tile_off, int64_t n_gb, int64_t w,
                                                  const RunWeights& rw, int lane) {
  int64_t lo = 0, hi = n_gb + 1;  // W(lo) <= w; the run holding weight w lies in [lo, hi)
  while (hi - lo > 1) {
    const int64_t step = (hi - lo + 31) / 32;
    const int64_t i = lo + (int64_t)lane * step;
    const unsigned m = __ballot_sync(0xffffffffu, i < hi && rw.start(tile_off, i) <= w);
    const int64_t nlo = lo + (int64_t)(31 - __clz(m)) * step;  // bit 0 is set: W(lo) <= w
    hi = min(hi, nlo + step);
    lo = nlo;
  }
  if (lo >= n_gb) return tile_off[n_gb];
  const int64_t t0 = tile_off[lo], tr = (int64_t)tile_off[lo + 1] - t0;
  return t0 + max((int64_t)0, min(tr, w - rw.start(tile_off, lo) - rw.own(lo)));  // with the run's first tile
}

// K-major, 128B-swizzled operand whose 8-row atoms are `sbo` bytes apart.
__device__ __forceinline__ uint64_t umma_desc_kmajor_sbo(uint32_t saddr, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, %0;\n" ::"n"(kEpiWarps * 32) : "memory"); }
// Named barrier of the epilogue warpgroup that also ANDs a flag over its threads.
__device__ __forceinline__ bool epi_bar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, 1, %2, p;\nselp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kEpiWarps * 32)
      : "memory");
  return r != 0;
}

// Named barrier of the two softmax warpgroups (id 2), plain and ANDing a flag.
__device__ __forceinline__ void soft_bar_sync() { asm volatile("bar.sync 2, %0;\n" ::"n"(2 * kSoftWarps * 32) : "memory"); }
__device__ __forceinline__ bool soft_bar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, 2, %2, p;\nselp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(2 * kSoftWarps * 32)
      : "memory");
  return r != 0;
}
// Per-warpgroup register budgets (all four warps of a warpgroup execute the
// same one).  512 threads launch with 128 registers each; the budgets after
// the split add up to the same 65536: producers 64, softmax 2 x 168, epilogue 112.
template <uint32_t N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(N)); }
template <uint32_t N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(N)); }
constexpr uint32_t kRegsProducers = 64, kRegsSoftmax = 168, kRegsEpilogue = 112;
static_assert(4 * 32 * kRegsProducers + 8 * 32 * kRegsSoftmax + 4 * 32 * kRegsEpilogue == 512 * 128,
              "register split must add up to the launch's registers");


// PPR = 8 / gs records (of 16 positions) per tile, a compile-time constant so
// that each group size gets its own straight-line code.
template <int D, int BK, int PPR>
__global__ void __launch_bounds__(kThreadsT, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_po,
                   const TileRecord* __restrict__ rec, const int32_t* __restrict__ tile_off, int64_t max_tiles,
                   int H_q, int H_kv, int k, int64_t nb, int64_t T0, int64_t T1, float scale_log2,
                   float2* __restrict__ part_ml, DeviceStatus* st) {
  using L = AttnLayout<D, BK>;
  constexpr int GS = 8 / PPR;                  // heads per group = rows per position
  constexpr int P = kTilePositions * PPR;      // positions per tile
  constexpr int GS_SHIFT = GS == 8 ? 3 : GS == 4 ? 2 : GS == 2 ? 1 : 0;
  constexpr int LANE_POS = (P + 31) / 32;      // positions per lane in the Q loader
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ TileRecord meta[kMeta * PPR];  // slot i: records [i PPR, (i + 1) PPR)
  __shared__ float ex_m[2][kRowsT], ex_l[2][kRowsT];  // softmax halves: row maxima and partial sums
  __shared__ int64_t range_s[2];                       // this CTA's tiles [range_s[0], range_s[1])

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
  auto meta_full = [&](int i) { return bar0 + 8u * (19 + i); };
  auto meta_empty = [&](int i) { return bar0 + 8u * (19 + kMeta + i); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Rows of positions past a tile's count keep whatever an earlier tile left
  // there: zero the Q buffers once so that those rows of S stay finite.
  for (int i = tid; i < kQBufs * L::Q_BYTES / 16; i += kThreadsT)
    reinterpret_cast<uint4*>(smem + L::OFF_Q)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (tid == 0) {
    for (int i = 0; i < kQBufs; ++i) {
      mbar_init(q_full(i), 1);
      mbar_init(q_empty(i), 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(s_full(i), 1);
      mbar_init(p_full(i), 2 * kSoftWarps);
    }
    for (int i = 0; i < kOBufs; ++i) {
      mbar_init(o_full(i), 1);
      mbar_init(o_empty(i), kEpiWarps);
    }
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    mbar_init(drain_bar, 1);
    for (int i = 0; i < kMeta; ++i) {
      mbar_init(meta_full(i), 1);
      mbar_init(meta_empty(i), kMetaReaders);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == kWarpLoad) {
    // extra weight of a run start, in tiles (swept at 128K: 2 / 3 / 4 / 5 -> 16.82 / 16.53 / 16.57 / 16.62 ms
    // per attention call; a run before the slab: its K/V load only); with ppr > 1 a tile's own time dominates
    // and an equal count splits best
    const RunWeights rw{nb, min(nb, T0 / BK), min(nb, (T1 + BK - 1) / BK), PPR == 1 ? 3 : 0, PPR == 1 ? 1 : 0};
    const int64_t n_gb = (int64_t)H_kv * nb;
    const int64_t w_total = rw.start(tile_off, n_gb);
    const int64_t a = tile_at_weight(tile_off, n_gb, w_total * blockIdx.x / gridDim.x, rw, lane);
    const int64_t z = tile_at_weight(tile_off, n_gb, w_total * (blockIdx.x + 1) / gridDim.x, rw, lane);
    if (lane == 0) {
      range_s[0] = min(a, max_tiles);
      range_s[1] = min(z, max_tiles);
    }
  }
  if (warp == kWarpLoad && lane == 0) {
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
    prefetch_tmap(&tmap_po);
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&tmem_slot), L::TMEM_COLS);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;

  const int64_t t_begin = range_s[0];
  const int n = (int)(range_s[1] - range_s[0]);

  if (warp < kWarpSoft0) {
  regs_dec<kRegsProducers>();  // warps 0..3: the producers' warpgroup
  if (warp == kWarpMeta) {
    // ------------------------------------------------------------ tile records -> shared ring
    if (lane == 0) {
      bool ok = true;
      int issued = 0;
      for (int i = 0; i < n && ok; ++i) {
        const int ms_ = i % kMeta;
        if (!(ok = mbar_wait(meta_empty(ms_), ((i / kMeta) & 1) ^ 1, abort, st, 0x300))) break;
        mbar_arrive_expect_tx(meta_full(ms_), (uint32_t)(PPR * sizeof(TileRecord)));
        bulk_load(smem_u32(&meta[ms_ * PPR]), rec + (t_begin + i) * PPR, (uint32_t)(PPR * sizeof(TileRecord)),
                  meta_full(ms_));
        issued = i + 1;
      }
      // after an abort: wait for the copies still in flight before the CTA exits
      if (!ok)
        for (int i = max(0, issued - kMeta); i < issued; ++i)
          mbar_wait(meta_full(i % kMeta), (i / kMeta) & 1, nullptr, st, 0x3F1);
    }
  } else if (warp == kWarpLoad) {
    // ------------------------------------------------------------ Q loader
    bool ok = true;
    int issued = 0;
    for (int i = 0; i < n && ok; ++i) {
      const int ms_ = i % kMeta;
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(meta_full(ms_), (i / kMeta) & 1, abort, st, 0x400)))) break;
      const TileRecord* mt = &meta[ms_ * PPR];
      const int g = mt[0].g;
      int count = 0;
#pragma unroll
      for (int r = 0; r < PPR; ++r) count += mt[r].count;
      int32_t tl[LANE_POS];  // this lane's positions pp = lane + 32 j
#pragma unroll
      for (int j = 0; j < LANE_POS; ++j) {
        const int pp = lane + 32 * j;
        tl[j] = -1;
        if (pp < P && (pp & 15) < mt[pp >> 4].count) tl[j] = mt[pp >> 4].t[pp & 15];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(meta_empty(ms_));
      const int qb = i % kQBufs;
      int w = 1;
      if (lane == 0) {
        w = mbar_wait(q_empty(qb), ((i / kQBufs) & 1) ^ 1, abort, st, 0x401) ? 1 : 0;
        if (w) mbar_arrive_expect_tx(q_full(qb), (uint32_t)(count * L::NCD * GS * 128));
      }
      if (!(ok = __shfl_sync(0xffffffffu, w, 0) != 0)) break;
#pragma unroll
      for (int j = 0; j < LANE_POS; ++j) {
        const int pp = lane + 32 * j;
        if (tl[j] < 0) continue;
        // heads g*GS .. g*GS + GS - 1 of position tl[j] -> rows GS pp .. GS pp + GS - 1
        const uint32_t dst = sbase + L::OFF_Q + qb * L::Q_BYTES + (pp / PPR) * L::POS_BYTES + (pp % PPR) * GS * 128;
        if (GS == 8) {  // all d/64 atoms in one box
          tma_load_4d(dst, &tmap_q, 0, g * GS, 0, tl[j], q_full(qb));
        } else {        // one box of GS rows per atom
#pragma unroll
          for (int c = 0; c < L::NCD; ++c) tma_load_4d(dst + c * 1024, &tmap_q, 0, g * GS, c, tl[j], q_full(qb));
        }
      }
      issued = i + 1;
    }
    // after an abort: wait for the Q loads still in flight before the CTA exits
    if (!ok && lane == 0)
      for (int i = max(0, issued - kQBufs); i < issued; ++i)
        mbar_wait(q_full(i % kQBufs), (i / kQBufs) & 1, nullptr, st, 0x4F2);
  } else if (warp == kWarpKv) {
    // ------------------------------------------------------------ K/V loader
    if (lane == 0 && n > 0) {
      uint32_t runs = 0;
      int64_t prev = -1;
      int last = -1;
      bool ok = true;
      for (int i = 0; i < n && ok; ++i) {
        const int ms_ = i % kMeta;
        if (!(ok = mbar_wait(meta_full(ms_), (i / kMeta) & 1, abort, st, 0x403))) break;
        const int64_t gb = meta[ms_ * PPR].gb;
        const int g = meta[ms_ * PPR].g;
        const int32_t b = meta[ms_ * PPR].b;
        mbar_arrive(meta_empty(ms_));
        if (gb == prev) continue;
        prev = gb;
        if (!(ok = mbar_wait(kv_empty, (runs & 1) ^ 1, abort, st, 0x402))) break;
        mbar_arrive_expect_tx(kv_full, (uint32_t)(2 * L::K_BYTES));
        for (int c = 0; c < L::NCD; ++c) {
          tma_load_3d(sbase + L::OFF_K + c * L::KV_CHUNK, &tmap_k, c * 64, g, b * BK, kv_full);
          tma_load_3d(sbase + L::OFF_V + c * L::KV_CHUNK, &tmap_v, c * 64, g, b * BK, kv_full);
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
      // (g, b) of tile j from the record ring; the issuer holds a tile's slot
      // from its first look until that tile's P V has been issued
      int fetched = 0;
      auto gb_of = [&](int j, int32_t& out) -> bool {
        for (; fetched <= j; ++fetched)
          if (!mbar_wait(meta_full(fetched % kMeta), (fetched / kMeta) & 1, abort, st, 0x500)) return false;
        out = meta[(j % kMeta) * PPR].gb;
        return true;
      };
      int s_next = 0;  // next tile whose S is not issued
      int32_t gb_s_next = 0, gb_cur = 0;
      ok = gb_of(0, gb_s_next);
      auto issue_S = [&](int j, int64_t gb_j) -> bool {
        const int qb = j % kQBufs;
        if (!mbar_wait(q_full(qb), (j / kQBufs) & 1, abort, st, 0x501)) return false;
        if (gb_j != gb_staged) {
          if (!mbar_wait(kv_full, kv_cnt & 1, abort, st, 0x502)) return false;
          ++kv_cnt;
          gb_staged = gb_j;
        }
        tc_fence_after();
        // buffer j % 2 last held P(j-2), whose P V was issued before this S
        const uint32_t d = tmem + (uint32_t)((j % kSBufs) * 128);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int c = ks >> 2, kk = ks & 3;
          const uint64_t ad =
              umma_desc_kmajor_sbo(sbase + L::OFF_Q + qb * L::Q_BYTES + c * 1024 + kk * 32, L::POS_BYTES);
          const uint64_t bd = umma_desc_kmajor(sbase + L::OFF_K + c * L::KV_CHUNK + kk * 32, 128);
          mma_bf16_ss(d, ad, bd, IDESC_S, ks > 0);
        }
        umma_commit(s_full(j % kSBufs));
        umma_commit(q_empty(qb));
        return true;
      };
      for (int i = 0; i < n && ok; ++i) {
        if (!(ok = gb_of(i, gb_cur))) break;
        // S ahead: tile i+1 if it uses tile i's K/V block
        while (ok && s_next < n && s_next <= i + 1 && gb_s_next == gb_cur) {
          ok = issue_S(s_next, gb_s_next);
          ++s_next;
          if (ok && s_next < n) ok = gb_of(s_next, gb_s_next);
        }
        if (!ok) break;
        // PV(i)
        const int sb = i % kSBufs;
        if (!(ok = mbar_wait(p_full(sb), (i / kSBufs) & 1, abort, st, 0x503))) break;
        const int ob = i % kOBufs;
        if (!(ok = mbar_wait(o_empty(ob), ((i / kOBufs) & 1) ^ 1, abort, st, 0x504))) break;
        tc_fence_after();
        const uint32_t pcol = tmem + (uint32_t)(sb * 128);
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks) {
          // keys 16ks.. of half h = 16ks / (BK/2) sit packed at column h*BK/2 + (16ks - h*BK/2)/2
          constexpr int HW = BK / 2;
          const int h = (16 * ks) / HW;
          const uint32_t acol = pcol + (uint32_t)(h * HW + (16 * ks - h * HW) / 2);
          const uint64_t bd = umma_desc_mnmajor_sw128(sbase + L::OFF_V + ks * 16 * 128, L::KV_CHUNK);
          mma_bf16_ts(tmem + L::TMEM_O + (uint32_t)(ob * 128), acol, bd, IDESC_PV, ks > 0);
        }
        umma_commit(o_full(ob));
        mbar_arrive(meta_empty(i % kMeta));
        const bool last_of_block = (i + 1 == n) || (s_next > i + 1 ? false : gb_s_next != gb_cur);
        if (last_of_block) umma_commit(kv_empty);
      }
      if (!ok) {
        umma_commit(drain_bar);
        mbar_wait(drain_bar, 0, nullptr, st, 0x5F1);
      }
    }
  }
  } else if (warp < kWarpEpi0) {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax: both warpgroups on every tile
    // Warpgroup `half` owns key columns [half*HW, half*HW + HW) of every row
    // and writes its P (bf16, packed) over the first HW/2 of those columns.
    // The two halves exchange row maxima and partial sums through shared
    // memory at a named barrier of the eight warps.
    constexpr int HW = BK / 2;
    const int half = (warp - kWarpSoft0) / kSoftWarps;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int pos = row >> GS_SHIFT, hh = row & (GS - 1);
    const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
    for (int j = 0; j < n; ++j) {
      const int ms_ = j % kMeta;
      const bool w1 = mbar_wait(meta_full(ms_), (j / kMeta) & 1, abort, st, 0x600);
      const TileRecord& sr = meta[ms_ * PPR + (pos >> 4)];
      const int64_t t = (w1 && (pos & 15) < sr.count) ? sr.t[pos & 15] : -1;
      const int slot = sr.slot[pos & 15];
      const int tg = meta[ms_ * PPR].g;
      const int64_t tb = meta[ms_ * PPR].b;
      __syncwarp();
      if (lane == 0 && w1) mbar_arrive(meta_empty(ms_));
      const int sb = j % kSBufs;
      const uint32_t scol = tmem + lane_base + (uint32_t)(sb * 128 + half * HW);
      // Everything that does not need S is settled before waiting for it: the
      // row's partial (m, l) slot, and the last visible column of this half
      // (rows without output count as unmasked so that a warp takes the
      // masked path only where a real row needs it; TMEM loads are
      // warp-collective).
      const int64_t prow = t >= 0 ? ((t - T0) * k + slot) * H_q + (int64_t)tg * GS + hh : 0;
      const int64_t key0 = tb * BK + half * HW;
      const int lim = t < 0 ? HW - 1 : (int)max((int64_t)-1, min((int64_t)HW - 1, t - key0));
      const bool full = __all_sync(0xffffffffu, lim == HW - 1);
      const bool w2 = w1 && mbar_wait(s_full(sb), (j / kSBufs) & 1, abort, st, 0x601);
      // all eight warps leave together (the exchanges below are named barriers)
      if (!soft_bar_and(w2)) break;
      tc_fence_after();
      float m = __int_as_float(0xff800000);
      uint32_t x[HW / 32][32];
      if (full) {
#pragma unroll
        for (int c = 0; c < HW / 32; ++c) tmem_ld_x32(scol + c * 32, x[c]);
        tmem_ld_wait();
        float mc[HW / 32];
#pragma unroll
        for (int c = 0; c < HW / 32; ++c) {
          mc[c] = __int_as_float(0xff800000);
#pragma unroll
          for (int e2 = 0; e2 < 32; e2 += 2) mc[c] = max3(mc[c], __uint_as_float(x[c][e2]), __uint_as_float(x[c][e2 + 1]));
        }
#pragma unroll
        for (int c = 0; c < HW / 32; ++c) m = fmaxf(m, mc[c]);
      } else {
        // diagonal tiles (and rows of blocks past t): masked, one chunk at a time
#pragma unroll 1
        for (int c = 0; c < HW / 32; ++c) {
          uint32_t y[32];
          tmem_ld_x32(scol + c * 32, y);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c * 32 + e <= lim) m = fmaxf(m, __uint_as_float(y[e]));
        }
      }
      ex_m[half][row] = m;
      soft_bar_sync();
      m = fmaxf(ex_m[0][row], ex_m[1][row]);
      const bool none = m == __int_as_float(0xff800000);
      const float ms = none ? 0.f : m * scale_log2;
      uint64_t lsum2 = 0;  // two fp32 zeros
      if (full) {
        const uint64_t nms2 = f2_pack(-ms, -ms);
#pragma unroll
        for (int c = 0; c < HW / 32; ++c) {
          uint32_t px[16];
#pragma unroll
          for (int e2 = 0; e2 < 32; e2 += 4) {
            float a0, a1, b0, b1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(x[c][e2]), __uint_as_float(x[c][e2 + 1])), scale2, nms2), a0,
                      a1);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(x[c][e2 + 2]), __uint_as_float(x[c][e2 + 3])), scale2, nms2),
                      b0, b1);
            a0 = ex2_approx(a0);
            a1 = ex2_approx(a1);
            b0 = ex2_approx(b0);
            b1 = ex2_approx(b1);
            lsum2 = f2_add(lsum2, f2_add(f2_pack(a0, a1), f2_pack(b0, b1)));
            px[e2 >> 1] = pack_bf16x2(a0, a1);
            px[(e2 >> 1) + 1] = pack_bf16x2(b0, b1);
          }
          tmem_st_x16(scol + c * 16, px);  // keys 32c..32c+31 of the half -> packed columns 16c..16c+15
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < HW / 32; ++c) {
          uint32_t y[32];
          tmem_ld_x32(scol + c * 32, y);
          tmem_ld_wait();
          uint32_t px[16];
          float l = 0.f;
#pragma unroll
          for (int e2 = 0; e2 < 32; e2 += 2) {
            float a0 = ex2_approx(fmaf(__uint_as_float(y[e2]), scale_log2, -ms));
            float a1 = ex2_approx(fmaf(__uint_as_float(y[e2 + 1]), scale_log2, -ms));
            a0 = c * 32 + e2 <= lim ? a0 : 0.f;
            a1 = c * 32 + e2 + 1 <= lim ? a1 : 0.f;
            l += a0 + a1;
            px[e2 >> 1] = pack_bf16x2(a0, a1);
          }
          lsum2 = f2_add(lsum2, f2_pack(l, 0.f));
          tmem_st_x16(scol + c * 16, px);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(sb));
      float l0, l1;
      f2_unpack(lsum2, l0, l1);
      ex_l[half][row] = l0 + l1;
      soft_bar_sync();
      // (m, l) of the row for the combine; m = -inf marks a row without keys
      if (half == 0 && t >= 0)
        part_ml[prow] = make_float2(none ? __int_as_float(0xff800000) : ms, ex_l[0][row] + ex_l[1][row]);
    }
  } else {
    regs_dec<kRegsEpilogue>();
    // ------------------------------------------------------------ epilogue warpgroup
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t ocol = tmem + ((uint32_t)(quarter * 32) << 16) + L::TMEM_O;
    const bool leader = warp == kWarpEpi0;
    const uint32_t stg = sbase + L::OFF_STG;
    // The staging tile is position-major: position p's block of SPB bytes holds
    // chunk c of head h in its row c * GS + h, so one TMA box {64, GS, d/64, 1}
    // stores the whole position.  Unit u of a row sits at u ^ (row address bits
    // 7..9) (the 128B swizzle).  With two chunks and GS < 8, lanes 4 apart would
    // share banks; those with lane bit 2 set walk their units in an order with
    // bit GS_SHIFT flipped, which keeps every quarter-warp's stores conflict-free.
    constexpr int SPB = L::NCD * GS * 128;
    constexpr uint32_t FLIP = (L::NCD == 2 && GS < 8) ? (1u << GS_SHIFT) : 0u;
    const bool flip = FLIP != 0 && ((lane >> 2) & 1);
    const uint32_t my_blk = stg + (uint32_t)((row >> GS_SHIFT) * SPB) + (uint32_t)(row & (GS - 1)) * 128;
    bool lead_ok = true;  // the store issuer's own waits
    for (int i = 0; i < n; ++i) {
      const int ob = i % kOBufs;
      const bool w = mbar_wait(o_full(ob), (i / kOBufs) & 1, abort, st, 0x701);
      // all four warps leave together (the named barriers have no time limit)
      if (!epi_bar_and(w && lead_ok)) break;
      tc_fence_after();
      // the whole row into registers as bf16 pairs, then O goes straight back to the tensor core
      uint32_t pk[D / 2];
#pragma unroll
      for (int c = 0; c < L::NCD; ++c) {
        uint32_t x[2][32];
        tmem_ld_x32(ocol + (uint32_t)(ob * 128) + c * 64, x[0]);
        tmem_ld_x32(ocol + (uint32_t)(ob * 128) + c * 64 + 32, x[1]);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e)
          pk[c * 32 + e] = pack_bf16x2(__uint_as_float(x[e >> 4][(e & 15) * 2]),
                                       __uint_as_float(x[e >> 4][(e & 15) * 2 + 1]));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty(ob));
      // the staging tile is free once the previous tile's stores have read it
      if (leader) bulk_wait_read_all();
      epi_bar_sync();
      // 16-byte unit u of 64-column chunk c -> its 128B-swizzled place in the row
#pragma unroll
      for (int c = 0; c < L::NCD; ++c) {
        const uint32_t ra = my_blk + (uint32_t)(c * GS * 128);
        const uint32_t xm = ((ra >> 7) & 7) ^ (flip ? FLIP : 0u);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int u0 = c * 32 + jj * 4, u1 = c * 32 + (jj ^ (int)FLIP) * 4;  // unit jj, or jj ^ FLIP
          const uint32_t a = ra + ((jj ^ xm) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(a), "r"(flip ? pk[u1] : pk[u0]),
                       "r"(flip ? pk[u1 + 1] : pk[u0 + 1]), "r"(flip ? pk[u1 + 2] : pk[u0 + 2]),
                       "r"(flip ? pk[u1 + 3] : pk[u0 + 3])
                       : "memory");
        }
      }
      fence_proxy_async_smem();
      epi_bar_sync();
      if (leader) {
        const int ms_ = i % kMeta;
        int w = 1;
        if (lane == 0) w = mbar_wait(meta_full(ms_), (i / kMeta) & 1, abort, st, 0x702) ? 1 : 0;
        lead_ok = __shfl_sync(0xffffffffu, w, 0) != 0;
        const TileRecord* mt = &meta[ms_ * PPR];
        if (lead_ok) {
          const int g = mt[0].g;
          bool any = false;
#pragma unroll
          for (int j = 0; j < LANE_POS; ++j) {
            const int pp = lane + 32 * j;
            if (pp >= P || (pp & 15) >= mt[pp >> 4].count) continue;
            const TileRecord& sr = mt[pp >> 4];
            const int32_t z = (int32_t)((sr.t[pp & 15] - T0) * k + sr.slot[pp & 15]);
            tma_store_4d(&tmap_po, stg + (uint32_t)(pp * SPB), 0, g * GS, 0, z);  // GS heads x d in one box
            any = true;
          }
          if (any) bulk_commit();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(meta_empty(ms_));
      }
    }
    if (leader) bulk_wait_all();
  }

  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int D, int BK, int PPR>
cudaError_t launch_t(const void* q, const void* kk, const void* vv, const TileRecord* rec, const int32_t* tile_off,
                     int64_t N, int H_q, int H_kv, int k, int64_t nb, int gs, int ppr, int64_t T0, int64_t T1,
                     int64_t rows,
                     int64_t max_tiles, float scale, uint16_t* part_o, float2* part_ml, DeviceStatus* st,
                     cudaStream_t s) {
  using L = AttnLayout<D, BK>;
  alignas(64) unsigned char tq[128], tk[128], tv[128], tpo[128];
  const uint64_t row_bytes = (uint64_t)D * 2;
  // Q and partial O as [rows][H_q][d/64][64] viewed in the order {64, H_q, d/64, rows}: a box
  // {64, heads, d/64, 1} lands as d/64 atoms of `heads` x 128 bytes, i.e. the tiles' layout.
  const uint64_t q_dims[4] = {64, (uint64_t)H_q, (uint64_t)L::NCD, (uint64_t)N};
  const uint64_t po_dims[4] = {64, (uint64_t)H_q, (uint64_t)L::NCD, (uint64_t)rows};
  const uint64_t qo_strides[3] = {row_bytes, 128, (uint64_t)H_q * row_bytes};
  const uint32_t q_box[4] = {64, (uint32_t)gs, gs == 8 ? (uint32_t)L::NCD : 1u, 1};
  const uint32_t po_box[4] = {64, (uint32_t)gs, (uint32_t)L::NCD, 1};
  if (!encode_tmap_4d(tq, q, q_dims, qo_strides, q_box, 128) ||
      !encode_tmap_3d(tk, kk, (uint64_t)D, (uint64_t)H_kv, (uint64_t)N, row_bytes, (uint64_t)H_kv * row_bytes, 64,
                      1, BK, 128) ||
      !encode_tmap_3d(tv, vv, (uint64_t)D, (uint64_t)H_kv, (uint64_t)N, row_bytes, (uint64_t)H_kv * row_bytes, 64,
                      1, BK, 128) ||
      !encode_tmap_4d(tpo, part_o, po_dims, qo_strides, po_box, 128))
    return cudaErrorInvalidValue;
  auto kern = attn_tc_kernel<D, BK, PPR>;
  const int smem = L::SMEM > 120 * 1024 ? L::SMEM : 120 * 1024;  // one CTA per SM: TMEM is never contended
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<num_sms(), kThreadsT, smem, s>>>(
      *reinterpret_cast<const CUtensorMap*>(tq), *reinterpret_cast<const CUtensorMap*>(tk),
      *reinterpret_cast<const CUtensorMap*>(tv), *reinterpret_cast<const CUtensorMap*>(tpo), rec, tile_off,
      max_tiles, H_q, H_kv, k, nb, T0, T1, scale * 1.4426950408889634f, part_ml, st);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_tiles(const void* q, const void* kk, const void* vv, const TileRecord* rec,
                              const int32_t* tile_off, int64_t N, int H_q, int H_kv, int d, int Bk, int k, int64_t nb,
                              int gs, int ppr, int64_t T0, int64_t T1, int64_t rows, int64_t max_tiles, float scale,
                              uint16_t* part_o, float2* part_ml, DeviceStatus* st, cudaStream_t s) {
  using Fn = cudaError_t (*)(const void*, const void*, const void*, const TileRecord*, const int32_t*, int64_t, int,
                            int, int, int64_t, int, int, int64_t, int64_t, int64_t, int64_t, float, uint16_t*,
                            float2*, DeviceStatus*, cudaStream_t);
  // [d == 128][Bk == 128][log2 ppr]
  static const Fn table[2][2][4] = {
      {{launch_t<64, 64, 1>, launch_t<64, 64, 2>, launch_t<64, 64, 4>, launch_t<64, 64, 8>},
       {launch_t<64, 128, 1>, launch_t<64, 128, 2>, launch_t<64, 128, 4>, launch_t<64, 128, 8>}},
      {{launch_t<128, 64, 1>, launch_t<128, 64, 2>, launch_t<128, 64, 4>, launch_t<128, 64, 8>},
       {launch_t<128, 128, 1>, launch_t<128, 128, 2>, launch_t<128, 128, 4>, launch_t<128, 128, 8>}}};
  const int lp = ppr == 1 ? 0 : ppr == 2 ? 1 : ppr == 4 ? 2 : 3;
  const Fn launch = table[d == 128][Bk == 128][lp];
  return launch(q, kk, vv, rec, tile_off, N, H_q, H_kv, k, nb, gs, ppr, T0, T1, rows, max_tiles, scale, part_o, part_ml,
                st, s);
}

}  // namespace msa
