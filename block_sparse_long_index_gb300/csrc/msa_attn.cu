// msa_sparse_attn_fwd: KV-outer block-sparse attention with an LSE combine.
//
// "MSA" study note 2-3 (O = Attn(q, K_{g,B}, V_{g,B})), 3-3 "Main Branch"
// (exact softmax over the selected support, per-head weights, group-shared
// blocks) and 3-5 (KV-outer execution over the reverse index, hot tiles
// pre-chunked across CTAs, two-phase combine); chipsbuilder "Funzionamento
// Delle Due Branch" (only causally visible tokens of the selected blocks).
//
// Steps per call:
//   1. B -> B* (msa_invert.cu): per (group, block) the ascending list of
//      entries t*k + slot.
//   2. Per query slab [T0, T1): for every (group, block) the sub-list of
//      entries with t in the slab (two binary searches, the list is sorted),
//      cut into tiles of 16 positions; an exclusive scan turns the tile
//      counts into a flat work list (hot blocks simply yield more tiles),
//      and one 128-byte record per tile lists its positions and slots.
//   3. Tile kernel (msa_attn_tile.cu, persistent, tcgen05): K_b and V_b are
//      staged in shared memory once per run of tiles of the same block and
//      shared by each tile's 16 positions x 8 head slots = 128 query rows
//      (gs of every 8 used); S = Q K_b^T and O = P V_b on tensor cores; the
//      causal mask applies only where b == local(t).  Each row writes its
//      un-normalised partial O (bf16) and its (m, l) (fp32) for its (t, slot).
//   4. Combine: per (t, h) the partials of the row's slots are merged:
//      M = max m_s, L = sum l_s 2^(m_s - M), out = sum O_s 2^(m_s - M) / L.
#include <math.h>

#include <algorithm>

#include "msa_common.cuh"

namespace msa {

namespace {

constexpr int kTilePos = kTilePositions;  // query positions per tile (x 8 head slots = 128 MMA rows)

// ---------------------------------------------------------------- schedule
// For each (g, b): [lo, hi) of the group's entry list with t in [T0, T1).
__global__ void sched_count_kernel(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ entries,
                                   int64_t N, int G, int k, int64_t nb, int64_t T0, int64_t T1, int P,
                                   int32_t* __restrict__ lo_out, int32_t* __restrict__ cnt_out,
                                   int32_t* __restrict__ tiles_out) {
  int64_t gb = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gb >= (int64_t)G * nb) return;
  int g = (int)(gb / nb);
  int64_t b = gb % nb;
  const int32_t* rp = row_ptr + (int64_t)g * (nb + 1);
  const int32_t* E = entries + (int64_t)g * N * k;
  int32_t a = rp[b], z = rp[b + 1];
  // first entry with t >= T0, first with t >= T1 (entries ascend in t)
  int32_t l = a, h = z;
  while (l < h) {
    int32_t m = l + ((h - l) >> 1);
    if ((int64_t)(E[m] / k) < T0) l = m + 1; else h = m;
  }
  int32_t lo = l;
  h = z;
  while (l < h) {
    int32_t m = l + ((h - l) >> 1);
    if ((int64_t)(E[m] / k) < T1) l = m + 1; else h = m;
  }
  int32_t cnt = l - lo;
  lo_out[gb] = lo;
  cnt_out[gb] = cnt;
  tiles_out[gb] = (cnt + P - 1) / P;
}

// Exclusive scan over n = G*nb tile counts (in place into off[0..n]); off[n] = total.
__global__ void __launch_bounds__(1024) sched_scan_kernel(const int32_t* __restrict__ tiles, int64_t n,
                                                          int32_t* __restrict__ off) {
  __shared__ int32_t warp_sums[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t per = (n + blockDim.x - 1) / blockDim.x;
  const int64_t lo = min((int64_t)tid * per, n), hi = min(lo + per, n);
  int32_t sum = 0;
  for (int64_t i = lo; i < hi; ++i) sum += tiles[i];
  int32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = warp_sums[lane];
    int32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_sums[lane] = wi - w;
  }
  __syncthreads();
  int32_t run = warp_sums[warp] + incl - sum;
  for (int64_t i = lo; i < hi; ++i) {
    int32_t x = tiles[i];
    off[i] = run;
    run += x;
  }
  if (tid == blockDim.x - 1) off[n] = run;
}

// The last index i in [0, n) with a[i] <= x, for a non-decreasing a with
// a[0] <= x: a 32-ary search by one warp (each step samples 32 points and
// narrows the range 32-fold), so 8192 lists take three dependent loads.
__device__ __forceinline__ int64_t warp_last_le(const int32_t* __restrict__ a, int64_t n, int64_t x, int lane) {
  int64_t lo = 0, hi = n;  // a[lo] <= x; the answer lies in [lo, hi)
  while (hi - lo > 1) {
    const int64_t step = (hi - lo + 31) / 32;
    const int64_t i = lo + (int64_t)lane * step;
    const unsigned m = __ballot_sync(0xffffffffu, i < hi && (int64_t)a[i] <= x);
    const int64_t nlo = lo + (int64_t)(31 - __clz(m)) * step;  // bit 0 is set: a[lo] <= x
    hi = min(hi, nlo + step);
    lo = nlo;
  }
  return lo;
}

// Records of the tiles: persistent CTAs, each over a contiguous range [a, z)
// of the tile list.  Warp 0 finds the (g, b) lists that hold the range's first
// and last tile; the warps then note, in shared memory, the (g, b) of every
// tile of the range (a warp per list, lanes over its tiles); finally every
// thread fills (tile, position) items, 16 PPR per tile, four items at a time
// with all their loads issued before any store.
constexpr int kRecThreads = 256;
constexpr int kRecUnroll = 4;
template <int PPR>
__global__ void __launch_bounds__(kRecThreads) tile_records_kernel(const int32_t* __restrict__ tile_off,
                                                                  const int32_t* __restrict__ lo,
                                                                  const int32_t* __restrict__ cnt,
                                                                  const int32_t* __restrict__ entries, int64_t N,
                                                                  int k, int64_t nb, int64_t n_gb, int64_t max_tiles,
                                                                  TileRecord* __restrict__ rec) {
  constexpr int P = kTilePositions * PPR;
  extern __shared__ int32_t tab[];  // (g, b) of each tile of this CTA's range
  __shared__ int64_t range_gb[2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t total = min((int64_t)tile_off[n_gb], max_tiles);
  const int64_t a = total * blockIdx.x / gridDim.x, z = total * (blockIdx.x + 1) / gridDim.x;
  if (a >= z) return;
  if (warp == 0) {
    const int64_t g0 = warp_last_le(tile_off, n_gb, a, lane);
    const int64_t g1 = warp_last_le(tile_off, n_gb, z - 1, lane);
    if (lane == 0) {
      range_gb[0] = g0;
      range_gb[1] = g1;
    }
  }
  __syncthreads();
  const int64_t g0 = range_gb[0], g1 = range_gb[1];
  for (int64_t gb = g0 + warp; gb <= g1; gb += kRecThreads / 32) {
    const int64_t f = max((int64_t)tile_off[gb], a), l = min((int64_t)tile_off[gb + 1], z);
    for (int64_t t = f + lane; t < l; t += 32) tab[t - a] = (int32_t)gb;
  }
  __syncthreads();
  const int items = (int)(z - a) * P;  // at most 8192 tiles of 128 positions per CTA
  for (int it0 = tid; it0 < items; it0 += kRecThreads * kRecUnroll) {
    int32_t gbv[kRecUnroll], first[kRecUnroll], ctot[kRecUnroll], e[kRecUnroll];
#pragma unroll
    for (int u = 0; u < kRecUnroll; ++u) {
      const int it = it0 + u * kRecThreads;
      const int tl = it / P, q = it % P;
      gbv[u] = it < items ? tab[tl] : 0;
      const int64_t gb = gbv[u];
      first[u] = lo[gb] + (int32_t)(a + tl - tile_off[gb]) * P;
      ctot[u] = min(P, lo[gb] + cnt[gb] - first[u]);
      e[u] = (it < items && q < ctot[u]) ? entries[(gb / nb) * N * k + first[u] + q] : -1;
    }
#pragma unroll
    for (int u = 0; u < kRecUnroll; ++u) {
      const int it = it0 + u * kRecThreads;
      if (it >= items) break;
      const int tl = it / P, q = it % P;
      const int sub = q / kTilePositions, pp = q % kTilePositions;
      TileRecord& r = rec[(a + tl) * PPR + sub];
      if (pp == 0) {
        r.gb = gbv[u];
        r.g = (int32_t)(gbv[u] / nb);
        r.b = (int32_t)(gbv[u] % nb);
        r.count = max(0, min(kTilePositions, ctot[u] - sub * kTilePositions));
      }
      const int32_t t = e[u] >= 0 ? e[u] / k : -1;
      r.t[pp] = t;
      r.slot[pp] = (uint8_t)(e[u] >= 0 ? e[u] - t * k : 0);
    }
  }
}

// Grid of the record kernel: enough CTAs that one CTA's table of tiles stays
// within 32 KB of shared memory.
static int64_t records_grid(int64_t max_tiles, int64_t& tab_bytes) {
  int64_t grid = (int64_t)num_sms() * 4;
  const int64_t need = ceil_div(max_tiles, 8192);
  if (grid < need) grid = need;
  if (grid < 1) grid = 1;
  tab_bytes = (ceil_div(max_tiles, grid) + 1) * 4;
  return grid;
}

// ---------------------------------------------------------------- combine
// Persistent CTAs of 256 threads, two per SM, each walking the slab's query
// positions t with a stride of the grid.  Per position the partials (k slots x
// H_q heads x d, contiguous) are read once, coalesced, with all k slot loads of
// a thread's (head, 8-column) item in flight together; the next position's
// (m, l) pairs and block ids are copied into the other half of a shared-memory
// double buffer (cp.async) while this position streams.  Slot s of group g
// contributes iff its id is in [0, nb) and not repeated by an earlier slot (the
// set counts each block once).  Partial s of head h holds O_s = sum_j p_j v_j
// with p_j = 2^(s_j - m_s) (s_j in log2 units) and l_s = sum_j p_j; then
// M = max m_s, w_s = 2^(m_s - M) / sum_s l_s 2^(m_s - M), out = sum_s w_s O_s,
// lse = ln 2 (M + log2 sum_s l_s 2^(m_s - M)); no contribution gives out = 0,
// lse = -inf.
constexpr int kCombineThreads = 256;
constexpr int kCombineSlots = 16;  // slot loads in flight per item

struct CombineSmem {
  size_t ml, bidx, cw, use, total;  // byte offsets of one buffer's parts and the total
  int nbuf;
};
inline CombineSmem combine_smem(int k, int H_q, int G) {
  CombineSmem c;
  const size_t ml = align_up((size_t)k * H_q * 8, 16), bi = align_up((size_t)G * k * 4, 16);
  const size_t cw = align_up((size_t)k * H_q * 4, 16), use = align_up((size_t)G * k, 16);
  c.nbuf = 2 * (ml + bi) + cw + use <= 160 * 1024 ? 2 : 1;
  c.ml = 0;
  c.bidx = c.nbuf * ml;
  c.cw = c.bidx + c.nbuf * bi;
  c.use = c.cw + cw;
  c.total = c.use + use;
  return c;
}

__device__ __forceinline__ void cp_async_4(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_8(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kCombineThreads, 2) combine_kernel(
    const int32_t* __restrict__ block_idx, const uint16_t* __restrict__ part_o, const float2* __restrict__ part_ml,
    int64_t N, int H_q, int G, int gs, int k, int64_t nb, int64_t T0, int64_t rows, CombineSmem lay,
    uint16_t* __restrict__ out, float* __restrict__ lse) {
  extern __shared__ __align__(16) unsigned char cmb_s[];
  constexpr int C8 = D / 8;
  const int tid = threadIdx.x;
  const int kh = k * H_q, gk = G * k;
  float2* ml_s = reinterpret_cast<float2*>(cmb_s + lay.ml);      // [nbuf][k][H_q]
  int32_t* bidx_s = reinterpret_cast<int32_t*>(cmb_s + lay.bidx);  // [nbuf][G][k]
  float* cw = reinterpret_cast<float*>(cmb_s + lay.cw);            // [k][H_q] weights
  uint8_t* use_s = cmb_s + lay.use;                                // [G][k]
  const size_t ml_stride = (lay.bidx - lay.ml) / lay.nbuf / 8, bi_stride = (lay.cw - lay.bidx) / lay.nbuf / 4;
  auto fetch = [&](int64_t tr, int buf) {  // (m, l) and block ids of position T0 + tr into buffer buf
    const float2* pm = part_ml + tr * kh;
    for (int i = tid; i < kh; i += kCombineThreads) cp_async_8(ml_s + buf * ml_stride + i, pm + i);
    const int64_t t = T0 + tr;
    for (int i = tid; i < gk; i += kCombineThreads)
      cp_async_4(bidx_s + buf * bi_stride + i, block_idx + ((int64_t)(i / k) * N + t) * k + (i % k));
    cp_async_commit();
  };
  const int64_t stride = gridDim.x;
  int64_t tr = blockIdx.x;
  if (lay.nbuf == 2 && tr < rows) fetch(tr, 0);
  for (int it = 0; tr < rows; ++it, tr += stride) {
    const int buf = lay.nbuf == 2 ? (it & 1) : 0;
    const int64_t t = T0 + tr;
    const uint16_t* po = part_o + tr * kh * D;
    // the partial loads of this thread's first item do not need the weights: issue them first
    uint4 v[kCombineSlots];
    auto load_item = [&](int item, int s0) {
      const int h = item / C8, c8 = item % C8;
#pragma unroll
      for (int j = 0; j < kCombineSlots; ++j)
        if (s0 + j < k) v[j] = ldg_stream_16(po + ((int64_t)(s0 + j) * H_q + h) * D + c8 * 8);
    };
    if (tid < H_q * C8) load_item(tid, 0);
    if (lay.nbuf == 1) fetch(tr, 0);
    cp_async_wait<0>();
    __syncthreads();
    const float2* ml = ml_s + buf * ml_stride;
    const int32_t* bi = bidx_s + buf * bi_stride;
    for (int i = tid; i < gk; i += kCombineThreads) {  // slot s of group g counts iff valid and first of its id
      const int g = i / k, sl = i % k;
      const int32_t b = bi[i];
      bool ok = b >= 0 && (int64_t)b < nb;
      for (int s2 = 0; s2 < sl && ok; ++s2) ok = bi[g * k + s2] != b;
      use_s[i] = ok ? 1 : 0;
    }
    __syncthreads();
    if (lay.nbuf == 2 && tr + stride < rows) fetch(tr + stride, buf ^ 1);  // lands while this position streams
    for (int h = tid; h < H_q; h += kCombineThreads) {
      const uint8_t* use = use_s + (h / gs) * k;
      float M = __int_as_float(0xff800000);
      for (int sl = 0; sl < k; ++sl)
        if (use[sl]) M = fmaxf(M, ml[sl * H_q + h].x);
      float L = 0.f;
      for (int sl = 0; sl < k; ++sl) {
        const float e = use[sl] && M != __int_as_float(0xff800000) ? exp2f(ml[sl * H_q + h].x - M) : 0.f;
        cw[sl * H_q + h] = e;
        L += e * (use[sl] ? ml[sl * H_q + h].y : 0.f);
      }
      const float il = L > 0.f ? 1.f / L : 0.f;
      for (int sl = 0; sl < k; ++sl) cw[sl * H_q + h] *= il;
      lse[(int64_t)h * N + t] = L > 0.f ? (M + log2f(L)) * 0.69314718055994530942f : __int_as_float(0xff800000);
    }
    __syncthreads();
    for (int item = tid; item < H_q * C8; item += kCombineThreads) {
      const int h = item / C8, c8 = item % C8;
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.f;
      for (int s0 = 0; s0 < k; s0 += kCombineSlots) {
        if (item != tid || s0 != 0) load_item(item, s0);
#pragma unroll
        for (int j = 0; j < kCombineSlots; ++j) {
          if (s0 + j >= k) break;
          const float w = cw[(s0 + j) * H_q + h];
          // unused slots may hold stale bits: zero them instead of multiplying by w = 0
          const uint4 x = w != 0.f ? v[j] : make_uint4(0u, 0u, 0u, 0u);
          acc[0] = fmaf(w, bf16_lo(x.x), acc[0]);
          acc[1] = fmaf(w, bf16_hi(x.x), acc[1]);
          acc[2] = fmaf(w, bf16_lo(x.y), acc[2]);
          acc[3] = fmaf(w, bf16_hi(x.y), acc[3]);
          acc[4] = fmaf(w, bf16_lo(x.z), acc[4]);
          acc[5] = fmaf(w, bf16_hi(x.z), acc[5]);
          acc[6] = fmaf(w, bf16_lo(x.w), acc[6]);
          acc[7] = fmaf(w, bf16_hi(x.w), acc[7]);
        }
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(out + (t * H_q + h) * D + c8 * 8) = o;
    }
    __syncthreads();  // cw, use_s and this buffer are rewritten for the next position
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------- scratch layout
struct AttnScratch {
  int32_t *row_ptr, *entries, *n_entries;
  InvertScratch inv;
  int32_t *lo, *cnt, *tiles, *tile_off;
  TileRecord* rec;
  uint16_t* part_o;
  float2* part_ml;
};

static size_t carve(const AttnPlan& p, void* base, AttnScratch* out) {
  char* c = (char*)base;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* r = c ? c + off : nullptr;
    off += align_up(bytes, 256);
    return r;
  };
  const int G = p.H_kv;
  AttnScratch s;
  s.row_ptr = (int32_t*)take((size_t)G * (p.nb + 1) * 4);
  s.entries = (int32_t*)take((size_t)G * p.N * p.k * 4);
  s.n_entries = (int32_t*)take((size_t)G * 4);
  size_t inv_bytes = invert_scratch_bytes(p.N, G, p.Bk, p.k);
  char* inv_base = take(inv_bytes);
  s.inv = invert_scratch_carve(inv_base, p.N, G, p.Bk, p.k);
  s.lo = (int32_t*)take((size_t)G * p.nb * 4);
  s.cnt = (int32_t*)take((size_t)G * p.nb * 4);
  s.tiles = (int32_t*)take((size_t)G * p.nb * 4);
  s.tile_off = (int32_t*)take(((size_t)G * p.nb + 1) * 4);
  s.rec = (TileRecord*)take((size_t)p.max_tiles * p.ppr * sizeof(TileRecord));
  s.part_o = (uint16_t*)take((size_t)p.slab * p.k * p.H_q * p.d * 2);
  s.part_ml = (float2*)take((size_t)p.slab * p.k * p.H_q * 8);
  if (out) *out = s;
  return off;
}

}  // namespace

AttnPlan attn_plan(int64_t N, int H_q, int H_kv, int d, int Bk, int k) {
  AttnPlan p;
  p.N = N;
  p.H_q = H_q;
  p.H_kv = H_kv;
  p.d = d;
  p.Bk = Bk;
  p.k = k;
  p.gs = H_q / H_kv;
  p.nb = (N + Bk - 1) / Bk;
  // partial results of one slab: slab * k * H_q * (2d + 8) bytes, at most ~36 GB
  const double per_pos = (double)k * H_q * (2.0 * d + 8.0);
  int64_t cap = (int64_t)(36.0e9 / per_pos);
  if (cap > 131072) cap = 131072;
  if (cap < 1024) cap = 1024;
  p.slab = N < cap ? N : cap;
  p.ppr = 8 / p.gs;  // gs in {1, 2, 4, 8}
  // sum over (g, b) of ceil(cnt / P) <= entries / P + lists, P = 16 ppr positions per tile
  p.max_tiles = (int64_t)H_kv * ceil_div(p.slab * k, (int64_t)kTilePos * p.ppr) + (int64_t)H_kv * p.nb;
  return p;
}

size_t attn_scratch_bytes(const AttnPlan& p) { return carve(p, nullptr, nullptr); }

cudaError_t launch_tile_schedule(const int32_t* row_ptr, const int32_t* entries, int64_t N, int G, int k, int64_t nb,
                                 int64_t T0, int64_t T1, int64_t max_tiles, int ppr, int32_t* lo, int32_t* cnt,
                                 int32_t* tiles, int32_t* tile_off, TileRecord* rec, cudaStream_t s) {
  const int64_t n_gb = (int64_t)G * nb;
  sched_count_kernel<<<(unsigned)((n_gb + 255) / 256), 256, 0, s>>>(row_ptr, entries, N, G, k, nb, T0, T1,
                                                                    kTilePos * ppr, lo, cnt, tiles);
  sched_scan_kernel<<<1, 1024, 0, s>>>(tiles, n_gb, tile_off);
  int64_t tab_bytes = 0;
  const int64_t grid = records_grid(max_tiles, tab_bytes);
  auto rk = ppr == 1 ? tile_records_kernel<1> : ppr == 2 ? tile_records_kernel<2>
            : ppr == 4 ? tile_records_kernel<4> : tile_records_kernel<8>;
  rk<<<(unsigned)grid, kRecThreads, (size_t)tab_bytes, s>>>(tile_off, lo, cnt, entries, N, k, nb, n_gb, max_tiles,
                                                            rec);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                           int d_I, const AttnPlan& p, float scale, int32_t* block_idx, void* out, float* lse,
                           void* scratch, DeviceStatus* st, cudaStream_t s, bool f8, const int32_t* blk_lo) {
  cudaError_t e = launch_select(q_idx, k_idx, p.N, p.H_kv, d_I, p.Bk, p.k, block_idx, st, s, f8, blk_lo);
  if (e != cudaSuccess) return e;
  return launch_attn(q, k, v, block_idx, p, scale, out, lse, scratch, st, s);
}

cudaError_t launch_attn(const void* q, const void* k, const void* v, const int32_t* block_idx, const AttnPlan& p,
                        float scale, void* out, float* lse, void* scratch, DeviceStatus* st, cudaStream_t s) {
  AttnScratch sc;
  carve(p, scratch, &sc);
  const int G = p.H_kv;
  cudaError_t e = launch_invert(block_idx, p.N, G, p.Bk, p.k, sc.row_ptr, sc.entries, sc.n_entries, sc.inv, st, s);
  if (e != cudaSuccess) return e;
  for (int64_t T0 = 0; T0 < p.N; T0 += p.slab) {
    const int64_t T1 = T0 + p.slab < p.N ? T0 + p.slab : p.N;
    e = launch_tile_schedule(sc.row_ptr, sc.entries, p.N, G, p.k, p.nb, T0, T1, p.max_tiles, p.ppr, sc.lo, sc.cnt,
                             sc.tiles, sc.tile_off, sc.rec, s);
    if (e != cudaSuccess) return e;
    e = launch_attn_tiles(q, k, v, sc.rec, sc.tile_off, p.N, p.H_q, p.H_kv, p.d, p.Bk, p.k, p.nb, p.gs, p.ppr, T0,
                          T1, p.slab * p.k, p.max_tiles, scale, sc.part_o, sc.part_ml, st, s);
    if (e != cudaSuccess) return e;
    const CombineSmem lay = combine_smem(p.k, p.H_q, G);
    auto ck = p.d == 64 ? combine_kernel<64> : combine_kernel<128>;
    e = cudaFuncSetAttribute(ck, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lay.total);
    if (e != cudaSuccess) return e;
    const int64_t grid = std::min<int64_t>(T1 - T0, (int64_t)num_sms() * 2);
    ck<<<(unsigned)grid, kCombineThreads, lay.total, s>>>(block_idx, sc.part_o, sc.part_ml, p.N, p.H_q, G, p.gs, p.k,
                                                           p.nb, T0, T1 - T0, lay, (uint16_t*)out, lse);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace msa
