// msa_sparse_attn_bwd: gradients of block-sparse attention (main branch) and
// of the index branch's KL alignment loss.
//
// "MSA" study note 4-2 (the index branch is trained by a KL loss whose teacher
// is the mean of the GQA group's main-branch attention probabilities) and 4-3
// (the teacher is detached and the index input gets a stop-gradient, so the KL
// reaches only q^I and k^I); Flash-MSA "バックワードパス" (both backward passes
// run over the cached sparse blocks, scheduled through the inverted map B*,
// with the proxy LSE recomputed over the selected blocks) and "KLダイバージェ
// ンス損失" (the gradient on the proxy logits is the proxy probability minus the
// main probability).
//
// Per row (t, h), g = h / gs, J = the selected blocks' tokens j <= t:
//   P_j = exp(scale q.k_j - lse), D = dO.O, dZ_j = P_j (dO.v_j - D),
//   dq = scale sum_j dZ_j k_j, dk_j += scale dZ_j q, dv_j += P_j dO;
// per row (t, g): teacher pbar_j = mean_h P_j, index logits zI_j = q^I.k^I_j /
// sqrt(d_I), pI = softmax_J(zI), KL = sum_j pbar_j (log pbar_j - log pI_j),
//   dzI_j = w (pI_j - pbar_j), dq^I = sum_j dzI_j k^I_j / sqrt(d_I),
//   dk^I_j += dzI_j q^I / sqrt(d_I).
//
// Kernels, all over the forward's KV-outer tile list (B -> B*, tiles of 16
// positions x 8 head slots = 128 rows, one (group, block) per tile), built per
// query slab of at most 131072 positions (the slab bounds the teacher buffer;
// every gradient accumulates across slabs):
//   rowdot:     D[h, t] = dO.O;
//   index lse:  the masked index logits of each position over the tile's
//               block -> one (max, sum) per (t, slot); a combine per (t, g)
//               -> lse^I;
//   main:       S^T, P^T, dP^T, dZ^T of the tile's keys and rows; dV and dK
//               accumulated over the tiles of a (group, block) and flushed
//               with fp32 reductions; dQ added to dq with fp32 reductions
//               (TMA add-reductions from shared memory on tcgen05);
//               the teacher rows (mean P over each position's heads, bf16)
//               written per tile;
//   index:      the index logits again, dzI and the KL terms against the
//               teacher rows, dq^I added to dq_idx, dk^I accumulated over the
//               run.
// For d = Bk = d_I = 128 the three tile kernels run on tcgen05 (the *_tc
// kernels below: operands in 128B-swizzled shared memory, accumulators in
// TMEM, dK/dV and dk^I accumulated in TMEM across a run); other shapes use
// mma.sync kernels in which warps own 16-key slices and keep dK/dV in
// registers.  The tile kernels fetch the next tile's (or chunk's) rows and
// records while the current one computes.
// A block id repeated in a row's set contributes once (its first slot).
#include <math.h>

#include "msa_common.cuh"
#include "msa_sm100.cuh"
#include "msa_tiles.cuh"

namespace msa {

namespace {

using namespace tiles;

constexpr int kRowsT = 128;            // tile rows: kPosT positions x 8 head slots
constexpr int kPosT = kTilePositions;  // 16
constexpr int kThreadsB = 256;

// The contiguous range of the flat tile list this CTA walks.
// The CTAs split the tile list by weight, not by count: a (group, block) run
// weighs its tiles plus `rw` more for what its start costs (the K/V or K^I
// load, the dK/dV or dk^I flush at its end, its leading diagonal tiles, and in
// the index passes a partial chunk of 8 tiles).  With an equal count, per-CTA
// timers at 128K left the CTAs holding the late blocks' short runs 2 ms (main)
// and 3 ms (index gradient) behind the median.  The in-slab weights were swept
// at 128K (main/lse/gradient 0/0/0: 49.4 ms per call; 3/4/4: 46.6; 6/8/8: 46.2;
// 3/8/12: 45.2; 3/8/20: 45.4; 4/12/16: 45.4, flat around the chosen one).
// A slab's runs: n_gb = G nb runs in (group, block) order, r = g nb + b; the
// slab's own blocks are [b0, b1).  A run weighs its tiles plus `in` for its
// start when its block lies in the slab, `before` when the block precedes the
// slab (no diagonal tiles: later slabs of a long sequence), and 0 past the slab
// (no tiles).  The runs before r number g b0 + min(b, b0) before the slab and
// g (b1 - b0) + clamp(b - b0, 0, b1 - b0) inside it, so the prefix weight has a
// closed form and each warp finds its CTA's first and last tiles by a 32-ary
// search (every thread of the CTA calls tile_range, warp-uniformly).
struct RunSpan {
  int64_t n_gb, nb, b0, b1;
};
struct RunWeight {
  int64_t in, before;
};
constexpr RunWeight kRunWeightMain{3, 2}, kRunWeightLse{8, 7}, kRunWeightGrad{12, 11};
__device__ __forceinline__ int64_t run_start(const int32_t* __restrict__ tile_off, const RunSpan& rs, RunWeight rw,
                                             int64_t r) {
  const int64_t g = r / rs.nb, b = r % rs.nb;
  const int64_t before = g * rs.b0 + min(b, rs.b0);
  const int64_t in = g * (rs.b1 - rs.b0) + min(max(b - rs.b0, (int64_t)0), rs.b1 - rs.b0);
  return (int64_t)tile_off[r] + rw.before * before + rw.in * in;
}
__device__ __forceinline__ int64_t tile_at_weight(const int32_t* __restrict__ tile_off, const RunSpan& rs,
                                                  RunWeight rw, int64_t w) {
  const int lane = threadIdx.x & 31;
  int64_t lo = 0, hi = rs.n_gb + 1;  // W(lo) <= w; the run holding weight w lies in [lo, hi)
  while (hi - lo > 1) {
    const int64_t step = (hi - lo + 31) / 32;
    const int64_t i = lo + (int64_t)lane * step;
    const unsigned m = __ballot_sync(0xffffffffu, i < hi && run_start(tile_off, rs, rw, i) <= w);
    const int64_t nlo = lo + (int64_t)(31 - __clz(m)) * step;  // bit 0 is set: W(lo) <= w
    hi = min(hi, nlo + step);
    lo = nlo;
  }
  if (lo >= rs.n_gb) return tile_off[rs.n_gb];
  const int64_t b = lo % rs.nb, own = b < rs.b0 ? rw.before : b < rs.b1 ? rw.in : 0;
  const int64_t t0 = tile_off[lo], tr = (int64_t)tile_off[lo + 1] - t0;
  return t0 + max((int64_t)0, min(tr, w - run_start(tile_off, rs, rw, lo) - own));  // with the run's first tile
}
__device__ __forceinline__ void tile_range(const int32_t* tile_off, const RunSpan& rs, RunWeight rw, int64_t& lo,
                                           int64_t& hi) {
  const int64_t wt = run_start(tile_off, rs, rw, rs.n_gb);
  lo = tile_at_weight(tile_off, rs, rw, wt * blockIdx.x / gridDim.x);
  hi = tile_at_weight(tile_off, rs, rw, wt * (blockIdx.x + 1) / gridDim.x);
}

// The teacher rows pass between kernels as bf16 (round to nearest even).
__device__ __forceinline__ uint16_t teacher_bf16(float x) { return (uint16_t)(pack_bf16x2(x, 0.f) & 0xffffu); }
__device__ __forceinline__ float teacher_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

__device__ __forceinline__ void cp_async_4(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}

// Position t of row r of a tile (p = r / 8, head slot r % 8), or -1 past the
// tile's count or past gs (and for slots marked as repeats, see mark_repeats).
__device__ __forceinline__ int32_t row_t(const TileRecord& rc, int r, int gs) {
  const int p = r >> 3, hh = r & 7;
  return (p < rc.count && hh < gs) ? rc.t[p] : -1;
}

// Record ti of the list into a shared slot (eight 16-byte copies).
__device__ __forceinline__ void issue_record(TileRecord* slot, const TileRecord* rec, int64_t ti) {
  if (threadIdx.x < 8) cp_async_16(reinterpret_cast<char*>(slot) + 16 * threadIdx.x,
                                   reinterpret_cast<const char*>(rec + ti) + 16 * threadIdx.x, 16);
}

// A block id repeated in a row's set counts once: its later slots are marked
// t = -1 in the tile records, so the backward kernels skip them.
// With k a multiple of 4 a row's earlier slots are read as 16-byte pieces, all in flight before the compares.
__global__ void mark_repeats_kernel(TileRecord* __restrict__ rec, const int32_t* __restrict__ tile_off, int64_t n_gb,
                                    const int32_t* __restrict__ block_idx, int64_t N, int k) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t tile = i / kPosT;
  const int p = (int)(i % kPosT);
  if (tile >= tile_off[n_gb]) return;
  TileRecord& r = rec[tile];
  if (p >= r.count) return;
  const int32_t* sel = block_idx + ((int64_t)r.g * N + r.t[p]) * k;
  const int slot = r.slot[p];
  const int32_t b = r.b;
  bool rep = false;
  if ((k & 3) == 0) {
    int4 v[8];  // k <= 32
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 4 * j < slot ? __ldg(reinterpret_cast<const int4*>(sel) + j) : make_int4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      rep |= (4 * j < slot && v[j].x == b) || (4 * j + 1 < slot && v[j].y == b) || (4 * j + 2 < slot && v[j].z == b) ||
             (4 * j + 3 < slot && v[j].w == b);
  } else {
    for (int s2 = 0; s2 < slot && !rep; ++s2) rep = sel[s2] == b;
  }
  if (rep) r.t[p] = -1;
}

__device__ __forceinline__ void copy_record(TileRecord* dst, const TileRecord* src) {
  if (threadIdx.x < 8)
    reinterpret_cast<uint4*>(dst)[threadIdx.x] = __ldg(reinterpret_cast<const uint4*>(src) + threadIdx.x);
}

// ------------------------------------------------------------------ D = dO . O
// A row (t, h) is D/8 16-byte pieces, one per lane of a group of D/8 lanes;
// a warp takes 32 / (D/8) rows a step and kRowdotSteps steps, with every
// step's loads in flight before the sums.
constexpr int kRowdotSteps = 4;
template <int D>
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const uint16_t* __restrict__ dout,
                                                         const uint16_t* __restrict__ out, int64_t N, int H_q,
                                                         float* __restrict__ Dr) {
  constexpr int U = D / 8, RPS = 32 / U;  // lanes per row, rows per step
  const int lane = threadIdx.x & 31, u = lane % U;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t rows = N * H_q;
  const int64_t r0 = warp * (RPS * kRowdotSteps) + lane / U;  // t * H_q + h
  uint4 a[kRowdotSteps], b[kRowdotSteps];
#pragma unroll
  for (int j = 0; j < kRowdotSteps; ++j) {
    const int64_t row = r0 + (int64_t)j * RPS;
    const bool in = row < rows;
    a[j] = in ? ldg_stream_16(dout + row * D + 8 * u) : make_uint4(0u, 0u, 0u, 0u);
    b[j] = in ? ldg_stream_16(out + row * D + 8 * u) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int j = 0; j < kRowdotSteps; ++j) {
    const uint32_t x[4] = {a[j].x, a[j].y, a[j].z, a[j].w}, y[4] = {b[j].x, b[j].y, b[j].z, b[j].w};
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      s = fmaf(bf16_lo(x[e]), bf16_lo(y[e]), s);
      s = fmaf(bf16_hi(x[e]), bf16_hi(y[e]), s);
    }
#pragma unroll
    for (int o = U / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const int64_t row = r0 + (int64_t)j * RPS;
    if (u == 0 && row < rows) Dr[(row % H_q) * N + row / H_q] = s;
  }
}

// ------------------------------------------------------------------ index-branch lse
// Per tile: zI = q^I.k^I_j / sqrt(d_I) of its positions over the block's keys
// j <= t; one (max, sum of exp) per (t, slot) into part[g, t, slot].
template <int BK, int DI>
__global__ void __launch_bounds__(kThreadsB) bwd_index_lse_kernel(
    const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ k_idx, const TileRecord* __restrict__ rec,
    const int32_t* __restrict__ tile_off, RunSpan rs, int64_t N, int G, int k, float sI,
    float2* __restrict__ part) {
  __shared__ __align__(128) uint16_t kIs[BK * DI];
  __shared__ __align__(128) uint16_t qIs[kPosT * DI];
  __shared__ float red_m[8][kPosT], red_l[8][kPosT];
  __shared__ __align__(16) TileRecord rc;
  constexpr int KSL = BK / 16;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g8 = lane >> 2, c4 = lane & 3;
  const uint32_t kIs_a = smem_u32(kIs), qIs_a = smem_u32(qIs);
  int64_t lo, hi;
  tile_range(tile_off, rs, kRunWeightLse, lo, hi);
  int cur_gb = -1;
  for (int64_t ti = lo; ti < hi; ++ti) {
    __syncthreads();
    copy_record(&rc, rec + ti);
    __syncthreads();
    if (rc.gb != cur_gb) {
      cur_gb = rc.gb;
      load_rows(kIs, BK, DI, k_idx, [&](int r) -> const uint16_t* {
        const int64_t j = (int64_t)rc.b * BK + r;
        return j < N ? k_idx + j * DI : nullptr;
      });
    }
    load_rows(qIs, kPosT, DI, q_idx, [&](int p) -> const uint16_t* {
      return p < rc.count && rc.t[p] >= 0 ? q_idx + ((int64_t)rc.t[p] * G + rc.g) * DI : nullptr;
    });
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    float zi[2][4] = {};
    if (warp < KSL) {
#pragma unroll
      for (int kk = 0; kk < DI; kk += 16) {
        uint32_t a[4], b[4];
        lds_a(a, kIs_a, warp * 16, kk, DI);
        lds_b_nk(b, qIs_a, 0, kk, DI);
        mma2(zi[0], zi[1], a, b);
      }
    }
    // element (key row g8 + 8 half, position nt * 8 + 2 c4 + e)
    float mx[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int p = nt * 8 + 2 * c4 + e;
        const int64_t t = p < rc.count ? rc.t[p] : -1;  // -1: no position, or a repeated block
        float m = __int_as_float(0xff800000);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int64_t j = (int64_t)rc.b * BK + warp * 16 + g8 + 8 * half;
          const bool ok = warp < KSL && j <= t;
          zi[nt][2 * half + e] = ok ? zi[nt][2 * half + e] * sI : __int_as_float(0xff800000);
          m = fmaxf(m, zi[nt][2 * half + e]);
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        mx[nt][e] = m;
      }
    if (g8 == 0)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) red_m[warp][nt * 8 + 2 * c4 + e] = mx[nt][e];
    __syncthreads();
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int p = nt * 8 + 2 * c4 + e;
        float M = __int_as_float(0xff800000);
        for (int w = 0; w < KSL; ++w) M = fmaxf(M, red_m[w][p]);
        float l = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const float z = zi[nt][2 * half + e];
          l += z == __int_as_float(0xff800000) ? 0.f : __expf(z - M);
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        mx[nt][e] = l;
      }
    if (g8 == 0)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) red_l[warp][nt * 8 + 2 * c4 + e] = mx[nt][e];
    __syncthreads();
    if (tid < rc.count && rc.t[tid] >= 0) {
      float M = __int_as_float(0xff800000), L = 0.f;
      for (int w = 0; w < KSL; ++w) M = fmaxf(M, red_m[w][tid]);
      for (int w = 0; w < KSL; ++w) L += red_l[w][tid];
      part[((int64_t)rc.g * N + rc.t[tid]) * k + rc.slot[tid]] = make_float2(M, L);
    }
  }
}

// lse^I[g, t] from the (max, sum) of the row's slots; a slot counts iff its id
// is in [0, nb) and first of its kind in the row.  A row is kp lanes (k
// rounded up to a power of two, k <= 32), lane s holding slot s: the first of
// a kind is the lowest lane of its match group, and the max and the sum are
// shuffle reductions within the kp lanes, so a warp takes 32 / kp rows with
// coalesced loads.
__global__ void bwd_index_lse_combine_kernel(const float2* __restrict__ part, const int32_t* __restrict__ block_idx,
                                             int64_t N, int G, int k, int64_t nb, int64_t T0, int64_t S,
                                             float* __restrict__ lseI) {
  int kp = 1;
  while (kp < k) kp <<= 1;
  const int lane = threadIdx.x & 31, sub = lane / kp, s = lane % kp;
  const int64_t w = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * (32 / kp) + sub;  // g * S + (t - T0)
  const bool row_in = w < (int64_t)G * S;
  const int64_t i = row_in ? (w / S) * N + T0 + w % S : 0;  // g * N + t
  const bool in = row_in && s < k;
  const int32_t id = in ? __ldg(block_idx + i * k + s) : -1;
  const float2 pm = in ? __ldg(part + i * k + s) : make_float2(__int_as_float(0xff800000), 0.f);
  const unsigned long long key = ((unsigned long long)(unsigned)sub << 32) | (unsigned)id;
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  const bool ok = in && id >= 0 && (int64_t)id < nb && __ffs(peers) - 1 == lane;
  float M = ok ? pm.x : __int_as_float(0xff800000);
  for (int o = kp / 2; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = ok && M != __int_as_float(0xff800000) && pm.x != __int_as_float(0xff800000) ? pm.y * __expf(pm.x - M)
                                                                                        : 0.f;
  for (int o = kp / 2; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  if (row_in && s == 0) lseI[i] = L > 0.f ? M + logf(L) : __int_as_float(0x7f800000);  // +inf: no index logit
}

// ------------------------------------------------------------------ main branch
// Shared memory: K and V rows of the current (group, block); two sets of the
// tile's Q and dO rows (the next tile's land while this one computes); dZ.
template <int D, int BK>
struct MainSmem {
  static constexpr int K = 0, V = BK * D * 2, Q = 2 * BK * D * 2, DO = Q + 2 * kRowsT * D * 2,
                       DZ = DO + 2 * kRowsT * D * 2;
  static constexpr int BYTES = DZ + kRowsT * BK * 2;
};

template <int D, int BK>
__global__ void __launch_bounds__(kThreadsB, 1) bwd_main_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ kc, const uint16_t* __restrict__ vc,
    const uint16_t* __restrict__ dout, const float* __restrict__ lse, const float* __restrict__ Dr,
    const TileRecord* __restrict__ rec, const int32_t* __restrict__ tile_off, RunSpan rs, int64_t N, int H_q,
    int H_kv, int gs, float scale, float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dv,
    uint16_t* __restrict__ pbar_g) {
  using L = MainSmem<D, BK>;
  extern __shared__ __align__(128) uint8_t smb[];
  uint16_t* Ks = reinterpret_cast<uint16_t*>(smb + L::K);
  uint16_t* Vs = reinterpret_cast<uint16_t*>(smb + L::V);
  uint16_t* dZs = reinterpret_cast<uint16_t*>(smb + L::DZ);
  __shared__ float lse_s[2][kRowsT], D_s[2][kRowsT];
  __shared__ int32_t tpos_s[2][kPosT];  // position of each of the tile's 16 positions (-1: none)
  __shared__ __align__(16) TileRecord rc_s[3];
  constexpr int KSL = BK / 16;   // key slices of 16
  constexpr int RG = 8 / KSL;    // row groups (1 or 2)
  constexpr int RPW = kRowsT / RG;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g8 = lane >> 2, c4 = lane & 3;
  const int ksl = warp % KSL, rg = warp / KSL;
  const float inv_gs = 1.f / (float)gs;
  const uint32_t Ks_a = smem_u32(Ks), Vs_a = smem_u32(Vs), dZs_a = smem_u32(dZs);
  auto Qs = [&](int b) { return reinterpret_cast<uint16_t*>(smb + L::Q + b * kRowsT * D * 2); };
  auto dOs = [&](int b) { return reinterpret_cast<uint16_t*>(smb + L::DO + b * kRowsT * D * 2); };
  float accK[D / 8][4], accV[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) accK[i][e] = accV[i][e] = 0.f;
  int cur_gb = -1, cur_g = 0, cur_b = 0;
  // dK and dV of this warp's 16 keys of the current block into dk, dv
  auto flush = [&]() {
    if (cur_gb < 0) return;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int64_t j = (int64_t)cur_b * BK + ksl * 16 + g8 + 8 * half;
      if (j < N) {
        float* pk = dk + (j * H_kv + cur_g) * D + 2 * c4;
        float* pv = dv + (j * H_kv + cur_g) * D + 2 * c4;
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) {
          red_add2(pk + nd * 8, scale * accK[nd][2 * half], scale * accK[nd][2 * half + 1]);
          red_add2(pv + nd * 8, accV[nd][2 * half], accV[nd][2 * half + 1]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) accK[i][e] = accV[i][e] = 0.f;
  };
  // the rows of tile ti (record in slot ti % 3) into buffer b: positions, lse, D, Q and dO, all asynchronous
  auto issue_rows = [&](int64_t ti, int b) {
    const TileRecord& rc = rc_s[ti % 3];
    const int g = rc.g;
    if (tid < kPosT) tpos_s[b][tid] = tid < rc.count ? rc.t[tid] : -1;
    for (int r = tid; r < kRowsT; r += blockDim.x) {
      const int32_t t = row_t(rc, r, gs);
      if (t >= 0) {
        const int64_t h = g * gs + (r & 7);
        cp_async_4(&lse_s[b][r], lse + h * N + t);
        cp_async_4(&D_s[b][r], Dr + h * N + t);
      } else {
        lse_s[b][r] = __int_as_float(0x7f800000);
        D_s[b][r] = 0.f;
      }
    }
    load_rows(Qs(b), kRowsT, D, q, [&](int r) -> const uint16_t* {
      const int32_t t = row_t(rc, r, gs);
      return t >= 0 ? q + ((int64_t)t * H_q + g * gs + (r & 7)) * D : nullptr;
    });
    load_rows(dOs(b), kRowsT, D, dout, [&](int r) -> const uint16_t* {
      const int32_t t = row_t(rc, r, gs);
      return t >= 0 ? dout + ((int64_t)t * H_q + g * gs + (r & 7)) * D : nullptr;
    });
  };
  int64_t lo, hi;
  tile_range(tile_off, rs, kRunWeightMain, lo, hi);
  if (lo < hi) {
    issue_record(&rc_s[lo % 3], rec, lo);
    if (lo + 1 < hi) issue_record(&rc_s[(lo + 1) % 3], rec, lo + 1);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    issue_rows(lo, 0);
    cp_async_commit();
  }
  for (int64_t ti = lo; ti < hi; ++ti) {
    const int buf = (int)((ti - lo) & 1);
    cp_async_wait<0>();  // this tile's rows and the next record
    __syncthreads();
    const TileRecord& rc = rc_s[ti % 3];
    if (rc.gb != cur_gb) {
      flush();
      cur_gb = rc.gb;
      cur_g = rc.g;
      cur_b = rc.b;
      const int64_t kv_row = (int64_t)H_kv * D;
      load_rows(Ks, BK, D, kc, [&](int r) -> const uint16_t* {
        const int64_t j = (int64_t)cur_b * BK + r;
        return j < N ? kc + j * kv_row + (int64_t)cur_g * D : nullptr;
      });
      load_rows(Vs, BK, D, vc, [&](int r) -> const uint16_t* {
        const int64_t j = (int64_t)cur_b * BK + r;
        return j < N ? vc + j * kv_row + (int64_t)cur_g * D : nullptr;
      });
      cp_async_commit();
      cp_async_wait<0>();
      __syncthreads();
    }
    // the next tile's rows and the record after it, while this tile computes
    if (ti + 2 < hi) issue_record(&rc_s[(ti + 2) % 3], rec, ti + 2);
    if (ti + 1 < hi) issue_rows(ti + 1, buf ^ 1);
    cp_async_commit();
    const uint32_t Qs_a = smem_u32(Qs(buf)), dOs_a = smem_u32(dOs(buf));
    // position of row r, or -1 (no position, a repeated block, or a head slot past gs)
    auto row_pos = [&](int r) -> int32_t { return (r & 7) < gs ? tpos_s[buf][r >> 3] : -1; };

    // ---- phase A: this warp's 16 keys against its rows, 16 rows (two positions) at a time
    const int key0 = ksl * 16;
    for (int rc0 = 0; rc0 < RPW; rc0 += 16) {
      const int row0 = rg * RPW + rc0;
      float s[2][4] = {}, dp[2][4] = {};
#pragma unroll
      for (int kk = 0; kk < D; kk += 16) {
        uint32_t a[4], b[4];
        lds_a(a, Ks_a, key0, kk, D);
        lds_b_nk(b, Qs_a, row0, kk, D);
        mma2(s[0], s[1], a, b);
        lds_a(a, Vs_a, key0, kk, D);
        lds_b_nk(b, dOs_a, row0, kk, D);
        mma2(dp[0], dp[1], a, b);
      }
      // element (key g8 + 8 half, row row0 + 8 nt + 2 c4 + e): P^T and dZ^T; n-tile nt = one position
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float tsum[2] = {0.f, 0.f};  // teacher: sum of P over the position's head slots
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int r = row0 + nt * 8 + 2 * c4 + e;
          const int32_t t = row_pos(r);
          const float ls = lse_s[buf][r], dd = D_s[buf][r];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int64_t j = (int64_t)cur_b * BK + key0 + g8 + 8 * half;
            float pv = 0.f, zv = 0.f;
            if (t >= 0 && j <= t) {
              pv = __expf(s[nt][2 * half + e] * scale - ls);
              zv = pv * (dp[nt][2 * half + e] - dd);
            }
            s[nt][2 * half + e] = pv;
            dp[nt][2 * half + e] = zv;
            tsum[half] += pv;
            st_bf16(dZs, r, key0 + g8 + 8 * half, BK, zv);
          }
        }
        if (pbar_g) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            tsum[half] += __shfl_xor_sync(0xffffffffu, tsum[half], 1);
            tsum[half] += __shfl_xor_sync(0xffffffffu, tsum[half], 2);
          }
          if (c4 == 0) {
            uint16_t* pb = pbar_g + (ti * kPosT + row0 / 8 + nt) * BK + key0 + g8;
            pb[0] = teacher_bf16(tsum[0] * inv_gs);
            pb[8] = teacher_bf16(tsum[1] * inv_gs);
          }
        }
      }
      uint32_t pa[4], za[4];
      c_to_a(pa, s[0], s[1]);
      c_to_a(za, dp[0], dp[1]);
#pragma unroll
      for (int nd = 0; nd < D / 8; nd += 2) {
        uint32_t b[4];
        lds_b_kn(b, dOs_a, row0, nd * 8, D);
        mma2(accV[nd], accV[nd + 1], pa, b);
        lds_b_kn(b, Qs_a, row0, nd * 8, D);
        mma2(accK[nd], accK[nd + 1], za, b);
      }
    }
    __syncthreads();  // dZ complete

    // ---- phase B: dQ of rows [16 warp, 16 warp + 16) = scale dZ K
    {
      const int r0 = warp * 16;
      float acc[D / 8][4];
#pragma unroll
      for (int i = 0; i < D / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < BK; kk += 16) {
        uint32_t a[4];
        lds_a(a, dZs_a, r0, kk, BK);
#pragma unroll
        for (int nd = 0; nd < D / 8; nd += 2) {
          uint32_t b[4];
          lds_b_kn(b, Ks_a, kk, nd * 8, D);
          mma2(acc[nd], acc[nd + 1], a, b);
        }
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int r = r0 + g8 + 8 * half;
        const int32_t t = row_pos(r);
        if (t >= 0) {
          float* p = dq + ((int64_t)t * H_q + cur_g * gs + (r & 7)) * D + 2 * c4;
#pragma unroll
          for (int nd = 0; nd < D / 8; ++nd)
            red_add2(p + nd * 8, scale * acc[nd][2 * half], scale * acc[nd][2 * half + 1]);
        }
      }
    }
  }
  flush();
}

// ------------------------------------------------------------------ index branch
// Shared memory: the block's index keys; two sets of the tile's index queries
// and teacher rows (from the main kernel); dzI.
template <int BK, int DI>
struct IndexSmem {
  static constexpr int KI = 0, QI = BK * DI * 2, PB = QI + 2 * kPosT * DI * 2, DZ = PB + 2 * kPosT * BK * 2;
  static constexpr int BYTES = DZ + kPosT * BK * 2;
};

template <int BK, int DI>
__global__ void __launch_bounds__(kThreadsB, 1) bwd_index_kernel(
    const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ k_idx, const float* __restrict__ lseI,
    const uint16_t* __restrict__ pbar_g, const TileRecord* __restrict__ rec, const int32_t* __restrict__ tile_off,
    RunSpan rs, int64_t N, int G, float sI, float w, float* __restrict__ dq_idx, float* __restrict__ dk_idx,
    float* __restrict__ kl) {
  using L = IndexSmem<BK, DI>;
  extern __shared__ __align__(128) uint8_t smb[];
  uint16_t* kIs = reinterpret_cast<uint16_t*>(smb + L::KI);
  uint16_t* dzs = reinterpret_cast<uint16_t*>(smb + L::DZ);
  __shared__ float lseI_s[2][kPosT];
  __shared__ int32_t tp_s[2][kPosT];
  __shared__ __align__(16) TileRecord rc_s[3];
  constexpr int KSL = BK / 16;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g8 = lane >> 2, c4 = lane & 3;
  const uint32_t kIs_a = smem_u32(kIs), dzs_a = smem_u32(dzs);
  auto qIs = [&](int b) { return reinterpret_cast<uint16_t*>(smb + L::QI + b * kPosT * DI * 2); };
  auto pbs = [&](int b) { return reinterpret_cast<uint16_t*>(smb + L::PB + b * kPosT * BK * 2); };
  float accI[DI / 8][4];
#pragma unroll
  for (int i = 0; i < DI / 8; ++i) accI[i][0] = accI[i][1] = accI[i][2] = accI[i][3] = 0.f;
  int cur_gb = -1, cur_g = 0, cur_b = 0;
  auto flush = [&]() {
    if (cur_gb < 0 || warp >= KSL) return;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int64_t j = (int64_t)cur_b * BK + warp * 16 + g8 + 8 * half;
      if (j < N) {
        float* p = dk_idx + j * DI + 2 * c4;
#pragma unroll
        for (int nd = 0; nd < DI / 8; ++nd) red_add2(p + nd * 8, sI * accI[nd][2 * half], sI * accI[nd][2 * half + 1]);
      }
    }
#pragma unroll
    for (int i = 0; i < DI / 8; ++i) accI[i][0] = accI[i][1] = accI[i][2] = accI[i][3] = 0.f;
  };
  auto issue_rows = [&](int64_t ti, int b) {
    const TileRecord& rc = rc_s[ti % 3];
    if (tid < kPosT) {
      const int32_t t = tid < rc.count ? rc.t[tid] : -1;
      tp_s[b][tid] = t;
      if (t >= 0) cp_async_4(&lseI_s[b][tid], lseI + (int64_t)rc.g * N + t);
      else lseI_s[b][tid] = __int_as_float(0x7f800000);
    }
    load_rows(qIs(b), kPosT, DI, q_idx, [&](int p) -> const uint16_t* {
      const int32_t t = p < rc.count ? rc.t[p] : -1;
      return t >= 0 ? q_idx + ((int64_t)t * G + rc.g) * DI : nullptr;
    });
    const uint16_t* src = pbar_g + ti * kPosT * BK;  // the teacher rows the main kernel wrote for this tile
    uint16_t* dst = pbs(b);
    for (int i = tid; i < kPosT * BK / 8; i += blockDim.x) cp_async_16(dst + 8 * i, src + 8 * i, 16);
  };
  int64_t lo, hi;
  tile_range(tile_off, rs, kRunWeightGrad, lo, hi);
  if (lo < hi) {
    issue_record(&rc_s[lo % 3], rec, lo);
    if (lo + 1 < hi) issue_record(&rc_s[(lo + 1) % 3], rec, lo + 1);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    issue_rows(lo, 0);
    cp_async_commit();
  }
  for (int64_t ti = lo; ti < hi; ++ti) {
    const int buf = (int)((ti - lo) & 1);
    cp_async_wait<0>();
    __syncthreads();
    const TileRecord& rc = rc_s[ti % 3];
    if (rc.gb != cur_gb) {
      flush();
      cur_gb = rc.gb;
      cur_g = rc.g;
      cur_b = rc.b;
      load_rows(kIs, BK, DI, k_idx, [&](int r) -> const uint16_t* {
        const int64_t j = (int64_t)cur_b * BK + r;
        return j < N ? k_idx + j * DI : nullptr;
      });
      cp_async_commit();
      cp_async_wait<0>();
      __syncthreads();
    }
    if (ti + 2 < hi) issue_record(&rc_s[(ti + 2) % 3], rec, ti + 2);
    if (ti + 1 < hi) issue_rows(ti + 1, buf ^ 1);
    cp_async_commit();
    const uint32_t qIs_a = smem_u32(qIs(buf));
    const uint16_t* pb_s = pbs(buf);

    // ---- index logits of this warp's 16 keys for the 16 positions, dzI and the KL terms
    if (warp < KSL) {
      const int key0 = warp * 16;
      float zi[2][4] = {};
#pragma unroll
      for (int kk = 0; kk < DI; kk += 16) {
        uint32_t a[4], b[4];
        lds_a(a, kIs_a, key0, kk, DI);
        lds_b_nk(b, qIs_a, 0, kk, DI);
        mma2(zi[0], zi[1], a, b);
      }
      float klp[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int p = nt * 8 + 2 * c4 + e;
          const int32_t t = tp_s[buf][p];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int key = key0 + g8 + 8 * half;
            const int64_t j = (int64_t)cur_b * BK + key;
            float dz = 0.f;
            if (t >= 0 && j <= t) {
              const float logp = zi[nt][2 * half + e] * sI - lseI_s[buf][p];
              const float pb = teacher_f32(pb_s[p * BK + key]);
              dz = w * (__expf(logp) - pb);
              if (pb > 0.f) klp[nt][e] += pb * (__logf(pb) - logp);
            }
            zi[nt][2 * half + e] = dz;
            st_bf16(dzs, p, key, BK, dz);
          }
        }
      if (kl) {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float x = klp[nt][e];
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
            const int p = nt * 8 + 2 * c4 + e;
            if (g8 == 0 && tp_s[buf][p] >= 0) atomicAdd(kl + (int64_t)cur_g * N + tp_s[buf][p], x);
          }
      }
      // dk^I of these keys += dzI^T q^I (k = the 16 positions)
      uint32_t za[4];
      c_to_a(za, zi[0], zi[1]);
#pragma unroll
      for (int nd = 0; nd < DI / 8; nd += 2) {
        uint32_t b[4];
        lds_b_kn(b, qIs_a, 0, nd * 8, DI);
        mma2(accI[nd], accI[nd + 1], za, b);
      }
    }
    __syncthreads();  // dzI complete

    // ---- dq^I (16 positions x d_I) = sI dzI kI: warp w takes columns [16 w, 16 w + 16)
    if (warp * 16 < DI) {
      float acc[2][4] = {};
#pragma unroll
      for (int kk = 0; kk < BK; kk += 16) {
        uint32_t a[4], b[4];
        lds_a(a, dzs_a, 0, kk, BK);
        lds_b_kn(b, kIs_a, kk, warp * 16, DI);
        mma2(acc[0], acc[1], a, b);
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int p = g8 + 8 * half;
        const int32_t t = tp_s[buf][p];
        if (t >= 0) {
          float* pp = dq_idx + ((int64_t)t * G + cur_g) * DI + warp * 16 + 2 * c4;
          red_add2(pp, sI * acc[0][2 * half], sI * acc[0][2 * half + 1]);
          red_add2(pp + 8, sI * acc[1][2 * half], sI * acc[1][2 * half + 1]);
        }
      }
    }
  }
  flush();
}

// ------------------------------------------------------------------ scratch and launch
struct BwdScratch {
  int32_t *row_ptr, *entries, *n_entries;
  InvertScratch inv;
  int32_t *lo, *cnt, *tiles, *tile_off;
  TileRecord* rec;
  float *Dr, *lseI;
  float2* partI;
  uint16_t* pbar;  // [slab tile][16 positions][Bk keys] bf16: the teacher, written by the main kernel
  int64_t max_tiles, nb, slab;
};

size_t carve(int64_t N, int H_q, int G, int Bk, int k, void* base, BwdScratch* out) {
  char* c = (char*)base;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* r = c ? c + off : nullptr;
    off += align_up(bytes, 256);
    return r;
  };
  BwdScratch s;
  s.nb = ceil_div(N, Bk);
  // the per-slab buffer: the teacher rows, G k Bk 2 bytes a position
  const double per_pos = (double)G * k * Bk * 2.0;
  int64_t cap = (int64_t)(32.0e9 / per_pos);
  if (cap > 131072) cap = 131072;
  if (cap < 1024) cap = 1024;
  s.slab = N < cap ? N : cap;
  s.max_tiles = (int64_t)G * ceil_div(s.slab * k, kPosT) + (int64_t)G * s.nb;
  s.row_ptr = (int32_t*)take((size_t)G * (s.nb + 1) * 4);
  s.entries = (int32_t*)take((size_t)G * N * k * 4);
  s.n_entries = (int32_t*)take((size_t)G * 4);
  char* inv_base = take(invert_scratch_bytes(N, G, Bk, k));
  s.inv = invert_scratch_carve(inv_base, N, G, Bk, k);
  s.lo = (int32_t*)take((size_t)G * s.nb * 4);
  s.cnt = (int32_t*)take((size_t)G * s.nb * 4);
  s.tiles = (int32_t*)take((size_t)G * s.nb * 4);
  s.tile_off = (int32_t*)take(((size_t)G * s.nb + 1) * 4);
  s.rec = (TileRecord*)take((size_t)s.max_tiles * sizeof(TileRecord));
  s.Dr = (float*)take((size_t)H_q * N * 4);
  s.lseI = (float*)take((size_t)G * N * 4);
  s.partI = (float2*)take((size_t)G * N * k * 8);
  s.pbar = (uint16_t*)take((size_t)s.max_tiles * kPosT * Bk * 2);
  if (out) *out = s;
  return off;
}


// ------------------------------------------------------------------ main, on tcgen05 (d = Bk = 128)
// The same tile work as bwd_main_kernel with every product on the 5th
// generation tensor cores.  Shared-memory tiles (128 rows x 128 bf16 each)
// are in the canonical 128B-swizzled K-major layout (two 64-column chunks of
// 16 KB, 8-row groups 1 KB apart), so one tile serves as a K-major operand of
// one product and an MN-major operand of another.  Per tile:
//   S^T = K Q^T and dP^T = V dO^T (M = keys, N = rows, K = d) into TMEM
//   columns 0-127 and 128-255;
//   both warpgroups (thread = key = TMEM lane; warpgroup h takes tile rows
//   64h..64h+63) form P^T and dZ^T = P^T (dP^T - D), write P^T (bf16) back
//   over the first half of their own S^T columns and dZ^T (bf16) to shared
//   memory as a K-major tile over the rows, and write the teacher (mean P
//   over each position's slots);
//   dV += P^T dO (P^T read from TMEM) and dK += dZ^T Q (dO, Q as MN-major B)
//   accumulate in TMEM columns 256-383 and 384-511 over the tiles of a
//   (group, block) run; dQ = dZ K (M = rows: dZ^T read as an MN-major A; K
//   as MN-major B) into columns 128-255 (dP^T is consumed by then; P^T in
//   columns 0-127 stays untouched until the next tile's S^T);
//   each thread stages 64 columns of its dQ row in shared memory, which the
//   TMA unit adds to dq (fp32 add-reductions of gs-head boxes, one per
//   position and 32 columns); at a run's end each thread adds 64 columns of
//   its key's dK and dV to dk and dv with fp32 vector reductions.
// Q and dO rows are double-buffered: tile i+1's rows arrive by cp.async (and
// its per-row position, lse and D into registers) while tile i computes.
// Warp 4 owns TMEM and its lane 0 issues the MMAs.  Phases are separated by
// CTA barriers and MMA completion mbarriers; every wait is bounded.

namespace tcb {
constexpr int kChunk = 128 * 128;  // one 64-column chunk of a 128-row tile, bytes
constexpr int kTile = 2 * kChunk;  // one 128 x 128 bf16 tile
constexpr int kK = 0, kV = kTile, kQ = 2 * kTile, kDO = 4 * kTile, kZT = 6 * kTile;  // Q, dO: two buffers each
constexpr int kBar = 7 * kTile;
constexpr int kBytes = 1024 + kBar + 64;
constexpr uint32_t kIdescSS = sm100::idesc_bf16_f32(128, 128);
constexpr uint32_t kIdescMnB = kIdescSS | (1u << 16);             // B MN-major
constexpr uint32_t kIdescMnAB = kIdescSS | (1u << 15) | (1u << 16);  // A and B MN-major
// byte offset of element (row r, column c) of a 128 x 128 bf16 tile
__device__ __forceinline__ uint32_t off(int r, int c) {
  return (uint32_t)((c >> 6) * kChunk + (r >> 3) * 1024 + (r & 7) * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) +
                    ((c & 7) << 1));
}
// rows [0, 128) of a tile from src(r) (nullptr: zeros), 16-byte cp.async copies
template <typename F>
__device__ __forceinline__ void load_tile(uint8_t* base, const uint16_t* any, F src) {
  for (int i = threadIdx.x; i < 128 * 16; i += blockDim.x) {
    const int r = i >> 4, c = (i & 15) * 8;
    const uint16_t* gp = src(r);
    cp_async_16(base + off(r, c), gp ? gp + c : any, gp ? 16 : 0);
  }
}
__device__ __forceinline__ void red_add4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
// fp32 add of a shared-memory box into the tensor behind `map` at {x, y, z}, by the TMA unit (bulk group)
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y,
                                                  int32_t z) {
  asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];\n" ::
                   "l"(reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// this thread's bulk operations have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
// ... and have completed
__device__ __forceinline__ void bulk_wait() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }
// fp32 add of `bytes` contiguous bytes of shared memory into global memory, by the TMA unit (bulk group);
// both addresses 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_reduce_add_f32(float* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;\n" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}
}  // namespace tcb

__global__ void __launch_bounds__(kThreadsB, 1) bwd_main_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_dq, const uint16_t* __restrict__ q, const uint16_t* __restrict__ kc, const uint16_t* __restrict__ vc,
    const uint16_t* __restrict__ dout, const float* __restrict__ lse, const float* __restrict__ Dr,
    const TileRecord* __restrict__ rec, const int32_t* __restrict__ tile_off, RunSpan rs, int64_t N, int H_q,
    int H_kv, int gs, float scale, float* __restrict__ dq, float* __restrict__ dk, float* __restrict__ dv,
    uint16_t* __restrict__ pbar_g, DeviceStatus* st) {
  using namespace tcb;
  constexpr int D = 128, BK = 128;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ __align__(16) float nlse2_s[kRowsT], nD_s[kRowsT];  // -lse in log2 units (-inf: no position), -D
  __shared__ int32_t trow_s[kRowsT];              // position of each tile row, -1 if none
  const uint32_t bar_s = sb + kBar, bar_q = sb + kBar + 8, bar_drain = sb + kBar + 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;  // TMEM lane quadrant, column half
  if (tid == 0) {
    sm100::mbar_init(bar_s, 1);
    sm100::mbar_init(bar_q, 1);
    sm100::mbar_init(bar_drain, 1);
    sm100::fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == 4) {
    sm100::tmem_alloc(smem_u32(&tmem_slot), 512);
    sm100::tc_fence_before();
  }
  __syncthreads();
  sm100::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;
  const float inv_gs = 1.f / (float)gs;
  const float kLog2e = 1.4426950408889634f;
  const int64_t kv_row = (int64_t)H_kv * D;
  int64_t lo, hi;
  tile_range(tile_off, rs, kRunWeightMain, lo, hi);
  // Rows of tile ti into Q/dO buffer b.  Thread tid copies 16-byte unit (tid & 15) of rows (tid >> 4) +
  // 16 m, m < 8: positions (tid >> 7) + 2 m, head slot (tid >> 4) & 7; the record fields it needs are
  // loaded together before any copy is issued.  The tile's (group, block) and the next tile's run key
  // are kept in registers for the loop.
  int32_t nx_gb = -1, nx_g = 0, nx_b = 0, nx2_gb = -1;
  auto issue_rows = [&](int64_t ti, int b) {
    const TileRecord* R = rec + ti;
    const int g = __ldg(&R->g), cnt = __ldg(&R->count);
    const int hs = (tid >> 4) & 7, p0 = tid >> 7, c = (tid & 15) * 8;
    int32_t tt[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) tt[m] = __ldg(&R->t[p0 + 2 * m]);
    nx_gb = __ldg(&R->gb);
    nx_b = __ldg(&R->b);
    nx2_gb = ti + 1 < hi ? __ldg(&rec[ti + 1].gb) : -1;
    nx_g = g;
    const bool slot_ok = hs < gs;
    const int64_t hrow = (int64_t)g * gs + hs;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const int r = (tid >> 4) + 16 * m;
      const int32_t t = (slot_ok && p0 + 2 * m < cnt) ? tt[m] : -1;
      const uint32_t o = off(r, c);
      const bool ok = t >= 0;
      cp_async_16(sm + kQ + b * kTile + o, ok ? q + ((int64_t)t * H_q + hrow) * D + c : q, ok ? 16 : 0);
      cp_async_16(sm + kDO + b * kTile + o, ok ? dout + ((int64_t)t * H_q + hrow) * D + c : dout, ok ? 16 : 0);
    }
  };
  // Row info of tile ti (thread tid < 128 = row tid): position, lse, D; loaded with the tile's rows (during
  // the previous tile), stored to shared memory at the tile's start.
  int32_t nt_t = -1;
  float nt_lse = 0.f, nt_D = 0.f;
  auto load_row_info = [&](int64_t ti) {
    if (tid < kRowsT) {
      const TileRecord* R = rec + ti;
      const int g = __ldg(&R->g), cnt = __ldg(&R->count);
      const int32_t tr = __ldg(&R->t[tid >> 3]);
      nt_t = ((tid & 7) < gs && (tid >> 3) < cnt) ? tr : -1;
      const int64_t h = (int64_t)g * gs + (tid & 7);
      nt_lse = nt_t >= 0 ? __ldg(&lse[h * N + nt_t]) : 0.f;
      nt_D = nt_t >= 0 ? __ldg(&Dr[h * N + nt_t]) : 0.f;
    }
  };
  if (lo < hi) {
    issue_rows(lo, 0);
    load_row_info(lo);
  }
  int32_t cur_gb = -1, cur_g = 0, cur_b = 0;
  uint32_t nt = 0;  // tiles done: the parity of both completion barriers
  bool issued = false;
  for (int64_t ti = lo; ti < hi; ++ti) {
    const int buf = (int)((ti - lo) & 1);
    const int32_t gb = nx_gb;
    const bool new_run = gb != cur_gb;
    const bool run_ends = ti + 1 >= hi || nx2_gb != gb;
    if (tid < kRowsT) {  // this tile's row info
      trow_s[tid] = nt_t;
      nlse2_s[tid] = nt_t >= 0 ? -nt_lse * kLog2e : -INFINITY;
      nD_s[tid] = -nt_D;
    }
    if (new_run) {
      cur_gb = gb;
      cur_g = nx_g;
      cur_b = nx_b;
      load_tile(sm + kK, kc, [&](int r) -> const uint16_t* {
        const int64_t j = (int64_t)cur_b * BK + r;
        return j < N ? kc + j * kv_row + (int64_t)cur_g * D : nullptr;
      });
      load_tile(sm + kV, vc, [&](int r) -> const uint16_t* {
        const int64_t j = (int64_t)cur_b * BK + r;
        return j < N ? vc + j * kv_row + (int64_t)cur_g * D : nullptr;
      });
    }
    cp_async_commit();
    cp_async_wait<0>();  // this tile's rows (issued during the previous tile) and a new run's K/V
    sm100::fence_proxy_async_smem();
    bulk_wait_read();  // the previous tile's dQ reductions have read their staging (buffer buf ^ 1)
    // full: every row either has no position or sees the whole block (t >= last key), so no key is masked
    const bool full =
        __syncthreads_and(tid >= kRowsT || nt_t < 0 || (int64_t)nt_t >= (int64_t)cur_b * BK + BK - 1) != 0;
    const uint32_t qb = sb + kQ + buf * kTile, dob = sb + kDO + buf * kTile;
    // ---- S^T and dP^T
    if (warp == 4 && lane == 0) {
      sm100::tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int c = ks >> 2, kk = ks & 3;
        sm100::mma_bf16_ss(tmem, sm100::umma_desc_kmajor(sb + kK + c * kChunk + kk * 32, 128),
                           sm100::umma_desc_kmajor(qb + c * kChunk + kk * 32, 128), kIdescSS, ks > 0);
        sm100::mma_bf16_ss(tmem + 128, sm100::umma_desc_kmajor(sb + kV + c * kChunk + kk * 32, 128),
                           sm100::umma_desc_kmajor(dob + c * kChunk + kk * 32, 128), kIdescSS, ks > 0);
      }
      sm100::umma_commit(bar_s);
      issued = true;
    }
    // the next tile's rows and row info stream in while this one computes (its buffer's last readers,
    // the previous tile's MMAs, have completed)
    if (ti + 1 < hi) {
      issue_rows(ti + 1, buf ^ 1);
      load_row_info(ti + 1);
    }
    cp_async_commit();
    // ---- P^T (to TMEM), dZ^T (to shared memory) and the teacher: thread = key
    if (sm100::mbar_wait(bar_s, nt & 1, abort, st, 0x801)) {
      sm100::tc_fence_after();
      const int key = quad * 32 + lane;
      const int64_t j = (int64_t)cur_b * BK + key;
      const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
      const float sl2 = scale * kLog2e;  // exp(x) = 2^(x log2 e)
      uint32_t sx[2][32], px[2][32];
      sm100::tmem_ld_x32(tmem + lane_base + half * 64, sx[0]);
      sm100::tmem_ld_x32(tmem + lane_base + 128 + half * 64, px[0]);
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {  // 32 rows at a time, the next 32 in flight
        const int cc = 2 * half + h2;
        sm100::tmem_ld_wait();
        sm100::reg_fence32(sx[h2]);
        sm100::reg_fence32(px[h2]);
        if (h2 == 0) {
          sm100::tmem_ld_x32(tmem + lane_base + half * 64 + 32, sx[1]);
          sm100::tmem_ld_x32(tmem + lane_base + 128 + half * 64 + 32, px[1]);
        }
        uint32_t pk[16], zk[16];
        float tsum[4] = {0.f, 0.f, 0.f, 0.f};
        if (full) {  // two rows per instruction; rows without a position get 2^-inf = 0
          const uint64_t sl2x2 = f2_pack(sl2, sl2);
          uint64_t tacc[4];
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) tacc[pp] = f2_pack(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 nl = *reinterpret_cast<const float4*>(&nlse2_s[cc * 32 + e]);
            const float4 nd = *reinterpret_cast<const float4*>(&nD_s[cc * 32 + e]);
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
              float a0, a1, z0, z1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(sx[h2][e + u]), __uint_as_float(sx[h2][e + u + 1])), sl2x2,
                               u ? f2_pack(nl.z, nl.w) : f2_pack(nl.x, nl.y)),
                        a0, a1);
              const float p0 = sm100::ex2_approx(a0), p1 = sm100::ex2_approx(a1);
              const uint64_t p2 = f2_pack(p0, p1);
              f2_unpack(f2_mul(p2, f2_add(f2_pack(__uint_as_float(px[h2][e + u]), __uint_as_float(px[h2][e + u + 1])),
                                          u ? f2_pack(nd.z, nd.w) : f2_pack(nd.x, nd.y))),
                        z0, z1);
              tacc[e >> 3] = f2_add(tacc[e >> 3], p2);
              pk[(e + u) >> 1] = pack_bf16x2(p0, p1);
              zk[(e + u) >> 1] = pack_bf16x2(z0, z1);
            }
          }
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) {
            float t0, t1;
            f2_unpack(tacc[pp], t0, t1);
            tsum[pp] = t0 + t1;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float pv[2], zv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int r = cc * 32 + e + u;
              const bool ok = j <= (int64_t)trow_s[r];  // -1 for rows without a position
              const float p = ok ? sm100::ex2_approx(fmaf(__uint_as_float(sx[h2][e + u]), sl2, nlse2_s[r])) : 0.f;
              pv[u] = p;
              zv[u] = p * (__uint_as_float(px[h2][e + u]) + nD_s[r]);
            }
            tsum[e >> 3] += pv[0] + pv[1];
            pk[e >> 1] = pack_bf16x2(pv[0], pv[1]);
            zk[e >> 1] = pack_bf16x2(zv[0], zv[1]);
          }
        }
        if (pbar_g) {
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) pbar_g[(ti * kPosT + cc * 4 + pp) * BK + key] = teacher_bf16(tsum[pp] * inv_gs);
        }
        // P^T rows 32 cc .. +31 -> packed columns 64 half + 16 h2 .. + 15 (within this warpgroup's S^T
        // columns, all already read)
        sm100::tmem_st_x16(tmem + lane_base + half * 64 + h2 * 16, pk);
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {  // 16-byte units: tile rows 32 cc + 8 q8 .. + 7
          const uint32_t o = off(key, cc * 32 + q8 * 8);
          *reinterpret_cast<uint4*>(sm + kZT + o) = make_uint4(zk[4 * q8], zk[4 * q8 + 1], zk[4 * q8 + 2], zk[4 * q8 + 3]);
        }
      }
      sm100::tmem_st_wait();
      sm100::fence_proxy_async_smem();
      sm100::tc_fence_before();
    }
    __syncthreads();
    if (*abort) break;
    // ---- dV, dK (accumulated over the run) and dQ
    if (warp == 4 && lane == 0) {
      sm100::tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kRowsT / 16; ++ks) {
        const int c = ks >> 2, kk = ks & 3;
        const uint32_t acc = (new_run && ks == 0) ? 0u : 1u;
        // P^T rows 16 ks .. : half h = ks / 4 holds them packed at columns 64 h + 8 (ks % 4)
        sm100::mma_bf16_ts(tmem + 256, tmem + (uint32_t)(64 * c + 8 * kk),
                           sm100::umma_desc_mnmajor_sw128(dob + ks * 16 * 128, kChunk), kIdescMnB, acc);
        sm100::mma_bf16_ss(tmem + 384, sm100::umma_desc_kmajor(sb + kZT + c * kChunk + kk * 32, 128),
                           sm100::umma_desc_mnmajor_sw128(qb + ks * 16 * 128, kChunk), kIdescMnB, acc);
      }
#pragma unroll
      for (int ks = 0; ks < BK / 16; ++ks)
        sm100::mma_bf16_ss(tmem + 128, sm100::umma_desc_mnmajor_sw128(sb + kZT + ks * 16 * 128, kChunk),
                           sm100::umma_desc_mnmajor_sw128(sb + kK + ks * 16 * 128, kChunk), kIdescMnAB, ks > 0);
      sm100::umma_commit(bar_q);
    }
    if (sm100::mbar_wait(bar_q, nt & 1, abort, st, 0x802)) {
      sm100::tc_fence_after();
      const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
      const int r = quad * 32 + lane;
      {  // dQ: thread = tile row r, warpgroup `half` = d columns 64 half .. + 63
        // The scaled rows are staged in this tile's Q (half 0) or dO (half 1) buffer, free now, as two
        // 32-column fp32 chunks of 128 rows x 128 bytes in the 128B-swizzled layout of the dq tensor map
        // (16-byte unit u of row r at u ^ (r % 8): conflict-free row-wise writes).  A position's gs rows are
        // one box {32 columns, gs heads, 1 position}; lanes 0-7 of each warp hand the warp's 4 positions x 2
        // chunks to the TMA unit as fp32 add-reductions into dq, which drain while the next tile computes.
        uint32_t x[2][32];
        sm100::tmem_ld_x32(tmem + lane_base + 128 + half * 64, x[0]);
        sm100::tmem_ld_x32(tmem + lane_base + 128 + half * 64 + 32, x[1]);
        sm100::tmem_ld_wait();
        const uint32_t stg = (half ? kDO : kQ) + buf * kTile;  // chunk j at stg + j kChunk
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint32_t* xs = &x[j][u * 4];
            *reinterpret_cast<float4*>(sm + stg + j * kChunk + r * 128 + ((u ^ (r & 7)) << 4)) =
                make_float4(scale * __uint_as_float(xs[0]), scale * __uint_as_float(xs[1]),
                            scale * __uint_as_float(xs[2]), scale * __uint_as_float(xs[3]));
          }
        sm100::fence_proxy_async_smem();
        __syncwarp();
        if (lane < 8) {
          const int p = quad * 4 + (lane >> 1), j = lane & 1;  // position of the tile, chunk of this half
          const int32_t t = trow_s[p * 8];
          if (t >= 0)
            tma_reduce_add_3d(&tmap_dq, sb + stg + j * kChunk + p * 1024, (2 * half + j) * 32, cur_g * gs, t);
          bulk_commit();
        }
      }
      if (run_ends) {  // thread = key: the run's dV and dK
        const int64_t j = (int64_t)cur_b * BK + r;
#pragma unroll 1
        for (int cc = 2 * half; cc < 2 * half + 2; ++cc) {
          uint32_t xv[32], xk[32];
          sm100::tmem_ld_x32(tmem + lane_base + 256 + cc * 32, xv);
          sm100::tmem_ld_x32(tmem + lane_base + 384 + cc * 32, xk);
          sm100::tmem_ld_wait();
          if (j < N) {
            float* pv = dv + (j * H_kv + cur_g) * D + cc * 32;
            float* pk2 = dk + (j * H_kv + cur_g) * D + cc * 32;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              red_add4(pv + e, __uint_as_float(xv[e]), __uint_as_float(xv[e + 1]), __uint_as_float(xv[e + 2]),
                       __uint_as_float(xv[e + 3]));
              red_add4(pk2 + e, scale * __uint_as_float(xk[e]), scale * __uint_as_float(xk[e + 1]),
                       scale * __uint_as_float(xk[e + 2]), scale * __uint_as_float(xk[e + 3]));
            }
          }
        }
      }
      sm100::tc_fence_before();
    }
    __syncthreads();
    if (*abort) break;
    ++nt;
  }
  cp_async_wait<0>();  // no copy of ours is left in flight when the CTA exits
  bulk_wait();
  __syncthreads();
  if (warp == 4) {
    if (lane == 0 && *abort && issued) {  // let the MMAs in flight finish before TMEM is released
      sm100::umma_commit(bar_drain);
      sm100::mbar_wait(bar_drain, 0, nullptr, st, 0x8F1);
    }
    __syncwarp();
    sm100::tc_fence_after();
    sm100::tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ index branch, on tcgen05 (Bk = d_I = 128)
// Both index-branch passes over chunks of up to 8 consecutive tiles of one
// (group, block) run: 128 positions, one per thread and TMEM lane (row r =
// 16 i + p is position p of the chunk's tile i; rows past the chunk are
// zero).  The index queries and the block's index keys are 128 x 128 bf16
// tiles in the 128B-swizzled K-major layout of the main kernel.
//   lse pass:  Z = Q^I K^I^T (M = positions, N = keys) into TMEM; each thread
//              reduces its row to one (max, sum of exp) per (t, slot);
//   gradient:  the same Z; each thread forms dzI = w (pI - pbar) of its row
//              and the row's KL terms, writes dzI (bf16) to shared memory;
//              dq^I = dzI K^I (K^I as MN-major B) over the Z columns, and
//              dk^I += dzI^T Q^I (dzI and Q^I read MN-major) accumulated in
//              TMEM columns 128-255 over the run's chunks, flushed with fp32
//              reductions at the run's end.
//              Each thread adds its dq^I row to dq_idx with one 512-byte bulk
//              fp32 add-reduction from shared memory.
// The lse pass needs 128 TMEM columns and 64 KB of shared memory (three CTAs
// per SM), the gradient pass 256 columns and 98 KB (two CTAs per SM); the
// CTAs of an SM overlap one another's loads and arithmetic.
namespace tci {
constexpr int kThreads = 128;
constexpr int kChunkTiles = 8;
constexpr int kRecs = kChunkTiles + 1;  // a chunk's records and the record after them (its run key)
constexpr int kKI = 0, kQI = tcb::kTile, kDZ = 2 * tcb::kTile;
constexpr int kLseBar = 2 * tcb::kTile, kLseBytes = 1024 + kLseBar + 64;
// the gradient pass stages its dq^I rows over the query and dzI tiles at a 528-byte row stride
constexpr int kStgRow = 528;
constexpr int kGradBar = kQI + 128 * kStgRow, kGradBytes = 1024 + kGradBar + 64;
constexpr uint32_t kIdescSS = tcb::kIdescSS, kIdescMnB = tcb::kIdescMnB, kIdescMnAB = tcb::kIdescMnAB;

// Records [ti0, ti0 + kRecs) that lie below hi into dst: 16-byte cp.async pieces, threads 0 .. 8 kRecs - 1.
__device__ __forceinline__ void fetch_records(TileRecord* dst, const TileRecord* rec, int64_t ti0, int64_t hi) {
  const int i = threadIdx.x >> 3;
  if (threadIdx.x < kRecs * 8 && ti0 + i < hi)
    cp_async_16(reinterpret_cast<char*>(dst) + 16 * threadIdx.x,
                reinterpret_cast<const char*>(rec + ti0) + 16 * threadIdx.x, 16);
}
struct Chunk {
  int n;          // tiles in the chunk
  bool run_ends;  // its (group, block) run ends with it, in this CTA's range
  int32_t gb;
  int g, b;
};
// The chunk starting at ti0 from its staged records: up to 8 tiles of one run.
__device__ __forceinline__ Chunk chunk_of(const TileRecord* RS, int64_t ti0, int64_t hi) {
  Chunk c;
  c.gb = RS[0].gb;
  c.g = RS[0].g;
  c.b = RS[0].b;
  int n = 1;
  while (n < kChunkTiles && ti0 + n < hi && RS[n].gb == c.gb) ++n;
  c.n = n;
  c.run_ends = ti0 + n >= hi || RS[n].gb != c.gb;
  return c;
}
// Position of chunk row r (tile r / 16, position r % 16), or -1 (no position, or a repeated block).
__device__ __forceinline__ int32_t row_t(const TileRecord* RS, int n, int r) {
  const int i = r >> 4, p = r & 15;
  return (i < n && p < RS[i].count) ? RS[i].t[p] : -1;
}
// Z = Q^I K^I^T: 8 steps over d_I.
__device__ __forceinline__ void issue_logits(uint32_t tmem, uint32_t sb) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const int c = ks >> 2, kk = ks & 3;
    sm100::mma_bf16_ss(tmem, sm100::umma_desc_kmajor(sb + kQI + c * tcb::kChunk + kk * 32, 128),
                       sm100::umma_desc_kmajor(sb + kKI + c * tcb::kChunk + kk * 32, 128), kIdescSS, ks > 0);
  }
}
// Copies of the run's index keys (new run) and the chunk's index queries into shared memory, and of the
// next chunk's records into the other record slot (a separate cp.async group, waited for at the next
// chunk).  Returns once the keys and queries have landed.
__device__ __forceinline__ void load_chunk(uint8_t* sm, const uint16_t* q_idx, const uint16_t* k_idx,
                                           const TileRecord* RS, const Chunk& ch, bool new_run, int G, int64_t N,
                                           TileRecord* next_slot, const TileRecord* rec, int64_t ti0, int64_t hi) {
  if (new_run)
    tcb::load_tile(sm + kKI, k_idx, [&](int r) -> const uint16_t* {
      const int64_t j = (int64_t)ch.b * 128 + r;
      return j < N ? k_idx + j * 128 : nullptr;
    });
  tcb::load_tile(sm + kQI, q_idx, [&](int r) -> const uint16_t* {
    const int32_t t = row_t(RS, ch.n, r);
    return t >= 0 ? q_idx + ((int64_t)t * G + ch.g) * 128 : nullptr;
  });
  cp_async_commit();
  if (ti0 + ch.n < hi) fetch_records(next_slot, rec, ti0 + ch.n, hi);
  cp_async_commit();
  cp_async_wait<1>();
  sm100::fence_proxy_async_smem();
}
}  // namespace tci

__global__ void __launch_bounds__(tci::kThreads, 3) bwd_index_lse_tc_kernel(
    const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ k_idx, const TileRecord* __restrict__ rec,
    const int32_t* __restrict__ tile_off, RunSpan rs, int64_t N, int G, int k, float sI,
    float2* __restrict__ part, DeviceStatus* st) {
  using namespace tci;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ __align__(16) TileRecord recs_s[2][kRecs];
  const uint32_t bar = sb + kLseBar, bar_drain = sb + kLseBar + 8;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    sm100::mbar_init(bar, 1);
    sm100::mbar_init(bar_drain, 1);
    sm100::fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == 0) {
    sm100::tmem_alloc(smem_u32(&tmem_slot), 128);
    sm100::tc_fence_before();
  }
  __syncthreads();
  sm100::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;
  const float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;
  const float s2 = sI * kLog2e;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  int64_t lo, hi;
  tile_range(tile_off, rs, kRunWeightLse, lo, hi);
  if (lo < hi) fetch_records(recs_s[0], rec, lo, hi);
  cp_async_commit();
  int32_t cur_gb = -1;
  uint32_t phase = 0;
  int slot = 0;
  bool issued = false;
  for (int64_t ti0 = lo; ti0 < hi;) {
    cp_async_wait<0>();  // this chunk's records
    __syncthreads();
    const TileRecord* RS = recs_s[slot];
    const Chunk ch = chunk_of(RS, ti0, hi);
    const int32_t t = row_t(RS, ch.n, tid);
    const int slot_k = t >= 0 ? (int)RS[tid >> 4].slot[tid & 15] : 0;
    load_chunk(sm, q_idx, k_idx, RS, ch, ch.gb != cur_gb, G, N, recs_s[slot ^ 1], rec, ti0, hi);
    cur_gb = ch.gb;
    __syncthreads();
    if (tid == 0) {
      sm100::tc_fence_after();
      issue_logits(tmem, sb);
      sm100::umma_commit(bar);
      issued = true;
    }
    if (sm100::mbar_wait(bar, phase & 1, abort, st, 0x803)) {
      sm100::tc_fence_after();
      const int64_t lim = (int64_t)t - (int64_t)ch.b * 128;  // keys c <= lim are visible to this row
      uint32_t x[4][32];
#pragma unroll
      for (int c32 = 0; c32 < 4; ++c32) sm100::tmem_ld_x32(tmem + lane_base + c32 * 32, x[c32]);
      sm100::tmem_ld_wait();
      float m = -INFINITY;  // base-2 units
      float l = 0.f;
      if (lim >= 127) {
        // every key visible (rows below the diagonal block): the maximum of the raw logits times s2 > 0 (the
        // rounding is monotonic, so it is the maximum of the scaled ones), then 2^(z s2 - m) by packed FMAs
        float mr[4];
#pragma unroll
        for (int c32 = 0; c32 < 4; ++c32) {
          mr[c32] = __uint_as_float(x[c32][0]);
#pragma unroll
          for (int e = 1; e < 31; e += 2)
            mr[c32] = sm100::max3(mr[c32], __uint_as_float(x[c32][e]), __uint_as_float(x[c32][e + 1]));
          mr[c32] = fmaxf(mr[c32], __uint_as_float(x[c32][31]));
        }
        m = fmaxf(fmaxf(mr[0], mr[1]), fmaxf(mr[2], mr[3])) * s2;
        const uint64_t s2x2 = f2_pack(s2, s2), nm2 = f2_pack(-m, -m);
        uint64_t acc = f2_pack(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          float a, b;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(x[c >> 5][c & 31]), __uint_as_float(x[c >> 5][(c & 31) + 1])),
                           s2x2, nm2),
                    a, b);
          acc = f2_add(acc, f2_pack(sm100::ex2_approx(a), sm100::ex2_approx(b)));
        }
        float l0, l1;
        f2_unpack(acc, l0, l1);
        l = l0 + l1;
      } else {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const float y = (c <= lim) ? __uint_as_float(x[c >> 5][c & 31]) * s2 : -INFINITY;
          x[c >> 5][c & 31] = __float_as_uint(y);
          m = fmaxf(m, y);
        }
        if (m > -INFINITY) {
#pragma unroll
          for (int c = 0; c < 128; ++c) l += sm100::ex2_approx(__uint_as_float(x[c >> 5][c & 31]) - m);
        }
      }
      if (t >= 0) part[((int64_t)ch.g * N + t) * k + slot_k] = make_float2(m > -INFINITY ? m * kLn2 : -INFINITY, l);
      sm100::tc_fence_before();
    }
    ++phase;
    __syncthreads();
    if (*abort) break;
    ti0 += ch.n;
    slot ^= 1;
  }
  cp_async_wait<0>();
  __syncthreads();
  if (warp == 0) {
    if ((tid & 31) == 0 && *abort && issued) {
      sm100::umma_commit(bar_drain);
      sm100::mbar_wait(bar_drain, 0, nullptr, st, 0x8F2);
    }
    __syncwarp();
    sm100::tc_fence_after();
    sm100::tmem_dealloc(tmem, 128);
  }
}

__global__ void __launch_bounds__(tci::kThreads, 2) bwd_index_tc_kernel(
    const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ k_idx, const float* __restrict__ lseI,
    const uint16_t* __restrict__ pbar_g, const TileRecord* __restrict__ rec, const int32_t* __restrict__ tile_off,
    RunSpan rs, int64_t N, int G, float sI, float w, float* __restrict__ dq_idx, float* __restrict__ dk_idx,
    float* __restrict__ kl, DeviceStatus* st) {
  using namespace tci;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ __align__(16) TileRecord recs_s[2][kRecs];
  const uint32_t bar = sb + kGradBar, bar_drain = sb + kGradBar + 8;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    sm100::mbar_init(bar, 1);
    sm100::mbar_init(bar_drain, 1);
    sm100::fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == 0) {
    sm100::tmem_alloc(smem_u32(&tmem_slot), 256);
    sm100::tc_fence_before();
  }
  __syncthreads();
  sm100::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;
  const float kLog2e = 1.4426950408889634f;
  const float s2 = sI * kLog2e;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  int64_t lo, hi;
  tile_range(tile_off, rs, kRunWeightGrad, lo, hi);
  if (lo < hi) fetch_records(recs_s[0], rec, lo, hi);
  cp_async_commit();
  int32_t cur_gb = -1;
  uint32_t phase = 0;
  int slot = 0;
  bool issued = false;
  for (int64_t ti0 = lo; ti0 < hi;) {
    cp_async_wait<0>();  // this chunk's records
    tcb::bulk_wait_read();  // the previous chunk's dq^I reductions have read their staging
    __syncthreads();
    const TileRecord* RS = recs_s[slot];
    const Chunk ch = chunk_of(RS, ti0, hi);
    const bool new_run = ch.gb != cur_gb;
    const int32_t t = row_t(RS, ch.n, tid);
    // this row's lse^I and teacher (the main kernel's row: tile ti0 + tid / 16, position tid % 16, 128
    // keys in bf16), requested before the copies so that all the latencies overlap
    const float lse_r = t >= 0 ? __ldg(&lseI[(int64_t)ch.g * N + t]) : INFINITY;
    const uint4* pb8 = reinterpret_cast<const uint4*>(pbar_g + ((ti0 + (tid >> 4)) * kPosT + (tid & 15)) * 128);
    uint4 pb[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) pb[e] = t >= 0 ? __ldg(pb8 + e) : make_uint4(0u, 0u, 0u, 0u);
    load_chunk(sm, q_idx, k_idx, RS, ch, new_run, G, N, recs_s[slot ^ 1], rec, ti0, hi);
    cur_gb = ch.gb;
    __syncthreads();
    if (tid == 0) {
      sm100::tc_fence_after();
      issue_logits(tmem, sb);
      sm100::umma_commit(bar);
      issued = true;
    }
    if (sm100::mbar_wait(bar, phase & 1, abort, st, 0x804)) {
      sm100::tc_fence_after();
      const int64_t lim = (int64_t)t - (int64_t)ch.b * 128;  // keys c <= lim are visible (none when t < 0)
      const float l2 = lse_r * kLog2e;
      float klsum = 0.f;
      const bool full = lim >= 127;  // rows below the diagonal block: every key visible
      const uint64_t s2x2 = f2_pack(s2, s2), nl2x2 = f2_pack(-l2, -l2), w2 = f2_pack(w, w), neg1 = f2_pack(-1.f, -1.f);
      uint64_t kl2 = f2_pack(0.f, 0.f);
      uint32_t x[2][32];
      sm100::tmem_ld_x32(tmem + lane_base, x[0]);
#pragma unroll
      for (int c32 = 0; c32 < 4; ++c32) {  // 32 keys at a time; the next 32 logits in flight
        sm100::tmem_ld_wait();
        sm100::reg_fence32(x[c32 & 1]);
        if (c32 < 3) sm100::tmem_ld_x32(tmem + lane_base + (c32 + 1) * 32, x[(c32 + 1) & 1]);
        uint32_t zk[16];
        if (full) {
          // every key visible: a pair of keys per packed instruction; the KL term of a key is
          // ln 2 * p (log2 p - log2 pI), with p = 0 contributing 0 (p times a finite log)
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const uint64_t y2 = f2_fma(f2_pack(__uint_as_float(x[c32 & 1][e]), __uint_as_float(x[c32 & 1][e + 1])),
                                       s2x2, nl2x2);  // log2 pI
            float y0, y1;
            f2_unpack(y2, y0, y1);
            const uint4& q8 = pb[c32 * 4 + (e >> 3)];
            const int cw = (e & 7) >> 1;
            const uint32_t wd = cw == 0 ? q8.x : cw == 1 ? q8.y : cw == 2 ? q8.z : q8.w;
            const float p0 = __uint_as_float(wd << 16), p1 = __uint_as_float(wd & 0xffff0000u);
            const uint64_t p2 = f2_pack(p0, p1);
            const uint64_t dz2 =
                f2_mul(w2, f2_add(f2_pack(sm100::ex2_approx(y0), sm100::ex2_approx(y1)), f2_mul(p2, neg1)));
            const uint64_t lp2 = f2_pack(lg2_approx(fmaxf(p0, 1e-30f)), lg2_approx(fmaxf(p1, 1e-30f)));
            kl2 = f2_fma(p2, f2_add(lp2, f2_mul(y2, neg1)), kl2);
            float d0, d1;
            f2_unpack(dz2, d0, d1);
            zk[e >> 1] = pack_bf16x2(d0, d1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float dz[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int c = c32 * 32 + e + u;
              const bool ok = c <= lim;
              const float y = fmaf(__uint_as_float(x[c32 & 1][e + u]), s2, -l2);  // log2 pI
              const uint4& q8 = pb[c32 * 4 + ((e + u) >> 3)];
              const int cc = (e + u) & 7;
              const uint32_t wd = (cc >> 1) == 0 ? q8.x : (cc >> 1) == 1 ? q8.y : (cc >> 1) == 2 ? q8.z : q8.w;
              const float p = __uint_as_float((cc & 1) ? (wd & 0xffff0000u) : (wd << 16));
              dz[u] = ok ? w * (sm100::ex2_approx(y) - p) : 0.f;
              if (ok && p > 0.f) klsum += p * (__logf(p) - y * 0.6931471805599453f);
            }
            zk[e >> 1] = pack_bf16x2(dz[0], dz[1]);
          }
        }
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          const uint32_t o = tcb::off(tid, c32 * 32 + q8 * 8);
          *reinterpret_cast<uint4*>(sm + kDZ + o) = make_uint4(zk[4 * q8], zk[4 * q8 + 1], zk[4 * q8 + 2], zk[4 * q8 + 3]);
        }
      }
      {
        float k0, k1;
        f2_unpack(kl2, k0, k1);
        klsum += 0.6931471805599453f * (k0 + k1);  // the full path's sum, in natural-log units
      }
      if (kl && t >= 0) atomicAdd(kl + (int64_t)ch.g * N + t, klsum);
      sm100::fence_proxy_async_smem();
      sm100::tc_fence_before();
    }
    ++phase;
    __syncthreads();
    if (*abort) break;
    if (tid == 0) {
      sm100::tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {  // dq^I = dzI K^I over the keys
        const int c = ks >> 2, kk = ks & 3;
        sm100::mma_bf16_ss(tmem, sm100::umma_desc_kmajor(sb + kDZ + c * tcb::kChunk + kk * 32, 128),
                           sm100::umma_desc_mnmajor_sw128(sb + kKI + ks * 16 * 128, tcb::kChunk), kIdescMnB, ks > 0);
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks)  // dk^I += dzI^T Q^I over the positions
        sm100::mma_bf16_ss(tmem + 128, sm100::umma_desc_mnmajor_sw128(sb + kDZ + ks * 16 * 128, tcb::kChunk),
                           sm100::umma_desc_mnmajor_sw128(sb + kQI + ks * 16 * 128, tcb::kChunk), kIdescMnAB,
                           (new_run && ks == 0) ? 0u : 1u);
      sm100::umma_commit(bar);
    }
    if (sm100::mbar_wait(bar, phase & 1, abort, st, 0x805)) {
      sm100::tc_fence_after();
      {  // thread = position: its dq^I row, staged over the (now free) query and dzI tiles at a 528-byte
         // stride (row-wise writes fall in distinct banks), then added to dq^I by one 512-byte bulk fp32
         // add-reduction, which drains while the next chunk loads and computes
        uint32_t x[4][32];
#pragma unroll
        for (int c32 = 0; c32 < 4; ++c32) sm100::tmem_ld_x32(tmem + lane_base + c32 * 32, x[c32]);
        sm100::tmem_ld_wait();
        uint8_t* row = sm + kQI + tid * kStgRow;
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const uint32_t* xs = &x[u >> 3][(u & 7) * 4];
          *reinterpret_cast<float4*>(row + u * 16) =
              make_float4(sI * __uint_as_float(xs[0]), sI * __uint_as_float(xs[1]), sI * __uint_as_float(xs[2]),
                          sI * __uint_as_float(xs[3]));
        }
        sm100::fence_proxy_async_smem();
        const int32_t tr = row_t(RS, ch.n, tid);
        if (tr >= 0) tcb::bulk_reduce_add_f32(dq_idx + ((int64_t)tr * G + ch.g) * 128, smem_u32(row), 512);
        tcb::bulk_commit();
      }
      if (ch.run_ends) {  // thread = key: the run's dk^I
        const int64_t j = (int64_t)ch.b * 128 + tid;
#pragma unroll 1
        for (int c32 = 0; c32 < 4; ++c32) {
          uint32_t x[32];
          sm100::tmem_ld_x32(tmem + lane_base + 128 + c32 * 32, x);
          sm100::tmem_ld_wait();
          if (j < N) {
            float* pk = dk_idx + j * 128 + c32 * 32;
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              tcb::red_add4(pk + e, sI * __uint_as_float(x[e]), sI * __uint_as_float(x[e + 1]),
                            sI * __uint_as_float(x[e + 2]), sI * __uint_as_float(x[e + 3]));
          }
        }
      }
      sm100::tc_fence_before();
    }
    ++phase;
    __syncthreads();
    if (*abort) break;
    ti0 += ch.n;
    slot ^= 1;
  }
  cp_async_wait<0>();
  tcb::bulk_wait();
  __syncthreads();
  if (warp == 0) {
    if ((tid & 31) == 0 && *abort && issued) {
      sm100::umma_commit(bar_drain);
      sm100::mbar_wait(bar_drain, 0, nullptr, st, 0x8F3);
    }
    __syncwarp();
    sm100::tc_fence_after();
    sm100::tmem_dealloc(tmem, 256);
  }
}

template <int D, int BK, int DI>
cudaError_t launch_tiles(const void* q, const void* kk, const void* v, const void* q_idx, const void* k_idx,
                         const int32_t* block_idx, const void* dout, const float* lse, const BwdScratch& sc,
                         int64_t N, int H_q, int H_kv, int k, float scale, float kl_weight, float* dq, float* dk,
                         float* dv, float* dq_idx, float* dk_idx, float* kl, int64_t T0, int64_t T1, DeviceStatus* st,
                         cudaStream_t s) {
  const int G = H_kv, gs = H_q / H_kv;
  const int64_t n_gb = (int64_t)G * sc.nb;
  const RunSpan rs{n_gb, sc.nb, T0 / BK, (T1 + BK - 1) / BK};
  const float sI = 1.f / sqrtf((float)DI);
  const int grid = num_sms();
  constexpr bool kIndexTc = BK == 128 && DI == 128;
  if constexpr (kIndexTc) {
    cudaError_t e0 = cudaFuncSetAttribute(bwd_index_lse_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          tci::kLseBytes);
    if (e0 != cudaSuccess) return e0;
    bwd_index_lse_tc_kernel<<<3 * grid, tci::kThreads, tci::kLseBytes, s>>>(
        (const uint16_t*)q_idx, (const uint16_t*)k_idx, sc.rec, sc.tile_off, rs, N, G, k, sI, sc.partI, st);
  } else {
    bwd_index_lse_kernel<BK, DI><<<grid, kThreadsB, 0, s>>>((const uint16_t*)q_idx, (const uint16_t*)k_idx, sc.rec,
                                                            sc.tile_off, rs, N, G, k, sI, sc.partI);
  }
  {
    int kp = 1;
    while (kp < k) kp <<= 1;
    const int64_t rows_per_cta = 8 * (32 / kp);  // 8 warps
    bwd_index_lse_combine_kernel<<<(unsigned)ceil_div((int64_t)G * (T1 - T0), rows_per_cta), 256, 0, s>>>(
        sc.partI, block_idx, N, G, k, sc.nb, T0, T1 - T0, sc.lseI);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if constexpr (D == 128 && BK == 128) {
    e = cudaFuncSetAttribute(bwd_main_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tcb::kBytes);
    if (e != cudaSuccess) return e;
    // dq as {d, H_q, N} fp32 with 32-column, gs-head boxes, 128B-swizzled: the main kernel's reductions
    alignas(64) unsigned char tdq[128];
    if (!encode_tmap_3d(tdq, dq, (uint64_t)D, (uint64_t)H_q, (uint64_t)N, (uint64_t)D * 4, (uint64_t)H_q * D * 4, 32,
                        (uint32_t)gs, 1, 128, 4))
      return cudaErrorInvalidValue;
    bwd_main_tc_kernel<<<grid, kThreadsB, tcb::kBytes, s>>>(*reinterpret_cast<const CUtensorMap*>(tdq),
                                                            (const uint16_t*)q, (const uint16_t*)kk,
                                                            (const uint16_t*)v, (const uint16_t*)dout, lse, sc.Dr,
                                                            sc.rec, sc.tile_off, rs, N, H_q, H_kv, gs, scale, dq,
                                                            dk, dv, sc.pbar, st);
  } else {
    auto km = bwd_main_kernel<D, BK>;
    e = cudaFuncSetAttribute(km, cudaFuncAttributeMaxDynamicSharedMemorySize, MainSmem<D, BK>::BYTES);
    if (e != cudaSuccess) return e;
    km<<<grid, kThreadsB, MainSmem<D, BK>::BYTES, s>>>((const uint16_t*)q, (const uint16_t*)kk, (const uint16_t*)v,
                                                      (const uint16_t*)dout, lse, sc.Dr, sc.rec, sc.tile_off, rs, N,
                                                      H_q, H_kv, gs, scale, dq, dk, dv, sc.pbar);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if constexpr (kIndexTc) {
    e = cudaFuncSetAttribute(bwd_index_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tci::kGradBytes);
    if (e != cudaSuccess) return e;
    bwd_index_tc_kernel<<<2 * grid, tci::kThreads, tci::kGradBytes, s>>>(
        (const uint16_t*)q_idx, (const uint16_t*)k_idx, sc.lseI, sc.pbar, sc.rec, sc.tile_off, rs, N, G, sI,
        kl_weight, dq_idx, dk_idx, kl, st);
    return cudaGetLastError();
  }
  auto ki = bwd_index_kernel<BK, DI>;
  e = cudaFuncSetAttribute(ki, cudaFuncAttributeMaxDynamicSharedMemorySize, IndexSmem<BK, DI>::BYTES);
  if (e != cudaSuccess) return e;
  ki<<<grid, kThreadsB, IndexSmem<BK, DI>::BYTES, s>>>((const uint16_t*)q_idx, (const uint16_t*)k_idx, sc.lseI,
                                                      sc.pbar, sc.rec, sc.tile_off, rs, N, G, sI, kl_weight, dq_idx,
                                                      dk_idx, kl);
  return cudaGetLastError();
}

template <int D, int BK>
cudaError_t launch_di(int d_I, const void* q, const void* kk, const void* v, const void* q_idx, const void* k_idx,
                      const int32_t* block_idx, const void* dout, const float* lse, const BwdScratch& sc, int64_t N,
                      int H_q, int H_kv, int k, float scale, float w, float* dq, float* dk, float* dv, float* dq_idx,
                      float* dk_idx, float* kl, int64_t T0, int64_t T1, DeviceStatus* st, cudaStream_t s) {
  if (d_I == 32)
    return launch_tiles<D, BK, 32>(q, kk, v, q_idx, k_idx, block_idx, dout, lse, sc, N, H_q, H_kv, k, scale, w, dq,
                                   dk, dv, dq_idx, dk_idx, kl, T0, T1, st, s);
  if (d_I == 64)
    return launch_tiles<D, BK, 64>(q, kk, v, q_idx, k_idx, block_idx, dout, lse, sc, N, H_q, H_kv, k, scale, w, dq,
                                   dk, dv, dq_idx, dk_idx, kl, T0, T1, st, s);
  return launch_tiles<D, BK, 128>(q, kk, v, q_idx, k_idx, block_idx, dout, lse, sc, N, H_q, H_kv, k, scale, w, dq,
                                  dk, dv, dq_idx, dk_idx, kl, T0, T1, st, s);
}

}  // namespace

size_t bwd_scratch_bytes(int64_t N, int H_q, int H_kv, int d, int Bk, int k) {
  (void)d;
  return carve(N, H_q, H_kv, Bk, k, nullptr, nullptr);
}

cudaError_t launch_bwd(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                       const int32_t* block_idx, const void* out, const float* lse, const void* dout, int64_t N,
                       int H_q, int H_kv, int d, int d_I, int Bk, int kb, float scale, float kl_weight, float* dq,
                       float* dk, float* dv, float* dq_idx, float* dk_idx, float* kl, void* scratch, DeviceStatus* st,
                       cudaStream_t s) {
  const int G = H_kv;
  BwdScratch sc;
  carve(N, H_q, G, Bk, kb, scratch, &sc);
  cudaError_t e;
  if ((e = cudaMemsetAsync(dq, 0, (size_t)N * H_q * d * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dk, 0, (size_t)N * H_kv * d * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dv, 0, (size_t)N * H_kv * d * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dq_idx, 0, (size_t)N * G * d_I * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dk_idx, 0, (size_t)N * d_I * 4, s)) != cudaSuccess) return e;
  if (kl && (e = cudaMemsetAsync(kl, 0, (size_t)G * N * 4, s)) != cudaSuccess) return e;
  if ((e = launch_invert(block_idx, N, G, Bk, kb, sc.row_ptr, sc.entries, sc.n_entries, sc.inv, st, s)) != cudaSuccess)
    return e;
  {
    const int64_t rows_per_cta = 8 * (32 / (d / 8)) * kRowdotSteps;  // 8 warps
    const unsigned grid = (unsigned)ceil_div(N * H_q, rows_per_cta);
    if (d == 64)
      bwd_rowdot_kernel<64><<<grid, 256, 0, s>>>((const uint16_t*)dout, (const uint16_t*)out, N, H_q, sc.Dr);
    else
      bwd_rowdot_kernel<128><<<grid, 256, 0, s>>>((const uint16_t*)dout, (const uint16_t*)out, N, H_q, sc.Dr);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // Query slabs [T0, T1) bound the teacher buffer; the gradients accumulate across slabs, and a slab's
  // positions have all their blocks in its tile list.
  for (int64_t T0 = 0; T0 < N; T0 += sc.slab) {
    const int64_t T1 = T0 + sc.slab < N ? T0 + sc.slab : N;
    if ((e = launch_tile_schedule(sc.row_ptr, sc.entries, N, G, kb, sc.nb, T0, T1, sc.max_tiles, 1, sc.lo, sc.cnt,
                                  sc.tiles, sc.tile_off, sc.rec, s)) != cudaSuccess)
      return e;
    mark_repeats_kernel<<<(unsigned)ceil_div(sc.max_tiles * kPosT, 256), 256, 0, s>>>(sc.rec, sc.tile_off,
                                                                                     (int64_t)G * sc.nb, block_idx, N,
                                                                                     kb);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (d == 64)
      e = Bk == 64 ? launch_di<64, 64>(d_I, q, k, v, q_idx, k_idx, block_idx, dout, lse, sc, N, H_q, H_kv, kb, scale,
                                       kl_weight, dq, dk, dv, dq_idx, dk_idx, kl, T0, T1, st, s)
                   : launch_di<64, 128>(d_I, q, k, v, q_idx, k_idx, block_idx, dout, lse, sc, N, H_q, H_kv, kb,
                                        scale, kl_weight, dq, dk, dv, dq_idx, dk_idx, kl, T0, T1, st, s);
    else
      e = Bk == 64 ? launch_di<128, 64>(d_I, q, k, v, q_idx, k_idx, block_idx, dout, lse, sc, N, H_q, H_kv, kb,
                                        scale, kl_weight, dq, dk, dv, dq_idx, dk_idx, kl, T0, T1, st, s)
                   : launch_di<128, 128>(d_I, q, k, v, q_idx, k_idx, block_idx, dout, lse, sc, N, H_q, H_kv, kb,
                                         scale, kl_weight, dq, dk, dv, dq_idx, dk_idx, kl, T0, T1, st, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace msa
