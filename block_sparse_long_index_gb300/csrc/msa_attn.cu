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
//      cut into tiles of P = 128 / gs positions; an exclusive scan turns the
//      tile counts into a flat work list (hot blocks simply yield more tiles).
//   3. Tile kernel (persistent): K_b and V_b are staged in shared memory once
//      per tile and shared by the tile's P positions x gs heads = 128 query
//      rows; S = Q K_b^T and O = P V_b on tensor cores; the causal mask
//      applies only where b == local(t).  Each row writes its normalised
//      partial O (bf16) and partial lse (fp32) for its (t, slot).
//   4. Combine: per (t, h) the partials of the row's slots are merged by their
//      lse into out and lse.
#include <math.h>

#include "msa_common.cuh"

namespace msa {

namespace {

constexpr int kTileRows = 128;
constexpr int kAttnThreads = 256;  // 8 warps x 16 rows

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

// ---------------------------------------------------------------- tile kernel
template <int D, int BK>
__global__ void __launch_bounds__(kAttnThreads) attn_tile_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ kk, const uint16_t* __restrict__ vv,
    const int32_t* __restrict__ entries, const int32_t* __restrict__ lo_arr, const int32_t* __restrict__ cnt_arr,
    const int32_t* __restrict__ tile_off, int64_t N, int H_q, int H_kv, int k, int64_t nb, int gs, int P,
    int64_t T0, float scale_log2, uint16_t* __restrict__ part_o, float* __restrict__ part_lse) {
  constexpr int LDS = D + 8;
  extern __shared__ __align__(16) uint16_t smem[];
  uint16_t* Qs = smem;                        // [128][LDS]
  uint16_t* Ks = Qs + kTileRows * LDS;        // [BK][LDS]
  uint16_t* Vs = Ks + BK * LDS;               // [BK][LDS]
  __shared__ int64_t pos_t[kTileRows];
  __shared__ int32_t pos_slot[kTileRows];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n_gb = (int64_t)H_kv * nb;
  const int32_t total = tile_off[n_gb];
  // a contiguous range of tiles per CTA: consecutive tiles mostly share (g, b), so K_b, V_b stay staged
  const int32_t t_begin = (int32_t)((int64_t)total * blockIdx.x / gridDim.x);
  const int32_t t_end = (int32_t)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  int64_t staged_gb = -1;

  for (int32_t tile = t_begin; tile < t_end; ++tile) {
    // locate (g, b) of this tile: largest gb with tile_off[gb] <= tile
    int64_t l = 0, h = n_gb;
    while (h - l > 1) {
      int64_t m = (l + h) >> 1;
      if (tile_off[m] <= tile) l = m; else h = m;
    }
    const int64_t gb = l;
    const int g = (int)(gb / nb);
    const int64_t b = gb % nb;
    const int32_t first = lo_arr[gb] + (tile - tile_off[gb]) * P;
    const int count = min(P, lo_arr[gb] + cnt_arr[gb] - first);
    const int32_t* E = entries + (int64_t)g * N * k;

    if (tid < P) {
      if (tid < count) {
        int32_t e = E[first + tid];
        pos_t[tid] = e / k;
        pos_slot[tid] = e % k;
      } else {
        pos_t[tid] = -1;
        pos_slot[tid] = 0;
      }
    }
    __syncthreads();

    // stage Q rows (row = p*gs + hh), K_b and V_b (rows past N are zero)
    for (int i = tid; i < kTileRows * (D / 8); i += kAttnThreads) {
      int r = i / (D / 8), c8 = i % (D / 8);
      int p = r / gs, hh = r % gs;
      int64_t t = (p < count) ? pos_t[p] : -1;
      const uint16_t* src = q + ((t < 0 ? 0 : t) * H_q + g * gs + hh) * D + c8 * 8;
      cp_async_16(Qs + r * LDS + c8 * 8, src, t < 0 ? 0 : 16);
    }
    if (gb != staged_gb) {
      for (int i = tid; i < BK * (D / 8); i += kAttnThreads) {
        int r = i / (D / 8), c8 = i % (D / 8);
        int64_t key = b * BK + r;
        bool ok = key < N;
        int64_t kc = ok ? key : 0;
        cp_async_16(Ks + r * LDS + c8 * 8, kk + (kc * H_kv + g) * D + c8 * 8, ok ? 16 : 0);
        cp_async_16(Vs + r * LDS + c8 * 8, vv + (kc * H_kv + g) * D + c8 * 8, ok ? 16 : 0);
      }
      staged_gb = gb;
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();

    // ---- S = Q K^T for this warp's 16 rows
    const int r_a = warp * 16 + (lane >> 2), r_b = r_a + 8;
    const int64_t t_a = (r_a / gs < count) ? pos_t[r_a / gs] : -1;
    const int64_t t_b = (r_b / gs < count) ? pos_t[r_b / gs] : -1;
    float s[BK / 8][4];
#pragma unroll
    for (int nt = 0; nt < BK / 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a[4];
      ldmatrix_x4(a[0], a[1], a[2], a[3], Qs + (warp * 16 + (lane & 15)) * LDS + ks * 16 + 8 * (lane >> 4));
#pragma unroll
      for (int np = 0; np < BK / 16; ++np) {
        uint32_t b0[2], b1[2];
        ldmatrix_x4(b0[0], b0[1], b1[0], b1[1],
                    Ks + (np * 16 + (lane & 7) + 8 * (lane >> 4)) * LDS + ks * 16 + 8 * ((lane >> 3) & 1));
        mma_bf16_16816(s[2 * np], a, b0);
        mma_bf16_16816(s[2 * np + 1], a, b1);
      }
    }
    // ---- causal mask (only the local block can hold keys past t) and softmax
    const int64_t key0 = b * BK;
    float m_a = __int_as_float(0xff800000), m_b = m_a;
#pragma unroll
    for (int nt = 0; nt < BK / 8; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        int64_t key = key0 + nt * 8 + 2 * (lane & 3) + e;
        if (key > t_a) s[nt][e] = __int_as_float(0xff800000);
        if (key > t_b) s[nt][2 + e] = __int_as_float(0xff800000);
        m_a = fmaxf(m_a, s[nt][e]);
        m_b = fmaxf(m_b, s[nt][2 + e]);
      }
    m_a = fmaxf(m_a, __shfl_xor_sync(0xffffffffu, m_a, 1));
    m_a = fmaxf(m_a, __shfl_xor_sync(0xffffffffu, m_a, 2));
    m_b = fmaxf(m_b, __shfl_xor_sync(0xffffffffu, m_b, 1));
    m_b = fmaxf(m_b, __shfl_xor_sync(0xffffffffu, m_b, 2));
    const bool empty_a = m_a == __int_as_float(0xff800000), empty_b = m_b == __int_as_float(0xff800000);
    const float ms_a = empty_a ? 0.f : m_a * scale_log2, ms_b = empty_b ? 0.f : m_b * scale_log2;
    float l_a = 0.f, l_b = 0.f;
#pragma unroll
    for (int nt = 0; nt < BK / 8; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float pa = exp2f(fmaf(s[nt][e], scale_log2, -ms_a));
        float pb = exp2f(fmaf(s[nt][2 + e], scale_log2, -ms_b));
        s[nt][e] = pa;
        s[nt][2 + e] = pb;
        l_a += pa;
        l_b += pb;
      }
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);

    // ---- O = P V
    float o[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[nt][e] = 0.f;
#pragma unroll
    for (int kb = 0; kb < BK / 16; ++kb) {
      uint32_t a[4];
      a[0] = pack_bf16x2(s[2 * kb][0], s[2 * kb][1]);
      a[1] = pack_bf16x2(s[2 * kb][2], s[2 * kb][3]);
      a[2] = pack_bf16x2(s[2 * kb + 1][0], s[2 * kb + 1][1]);
      a[3] = pack_bf16x2(s[2 * kb + 1][2], s[2 * kb + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t b0[2], b1[2];
        const int mat = lane >> 3;
        ldmatrix_x4_trans(b0[0], b0[1], b1[0], b1[1],
                          Vs + (kb * 16 + (lane & 7) + 8 * (mat & 1)) * LDS + dp * 16 + 8 * (mat >> 1));
        mma_bf16_16816(o[2 * dp], a, b0);
        mma_bf16_16816(o[2 * dp + 1], a, b1);
      }
    }

    // ---- normalised partial O (bf16) and partial lse (natural log)
    const float inv_a = empty_a ? 0.f : 1.f / l_a, inv_b = empty_b ? 0.f : 1.f / l_b;
    const float LN2 = 0.69314718055994530942f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = half ? r_b : r_a;
      const int p = r / gs, hh = r % gs;
      if (p >= count) continue;
      const int64_t t = pos_t[p];
      const int slot = pos_slot[p];
      const int hq = g * gs + hh;
      const int64_t prow = ((t - T0) * k + slot) * H_q + hq;
      const float inv = half ? inv_b : inv_a;
      uint16_t* dst = part_o + prow * D;
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        uint32_t w = pack_bf16x2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
        *reinterpret_cast<uint32_t*>(dst + nt * 8 + 2 * (lane & 3)) = w;
      }
      if ((lane & 3) == 0) {
        const bool empty = half ? empty_b : empty_a;
        const float ms = half ? ms_b : ms_a;
        const float l = half ? l_b : l_a;
        part_lse[prow] = empty ? __int_as_float(0xff800000) : (ms + log2f(l)) * LN2;
      }
    }
    __syncthreads();  // shared tiles are restaged by the next iteration
  }
}

// ---------------------------------------------------------------- combine
// One CTA per query position t: the position's partials (k slots x H_q heads x
// d, contiguous) are read once, coalesced.  Slot s of group g contributes iff
// its id is in [0, nb) and not repeated by an earlier slot (the set counts
// each block once).  out = sum_s w_s O_s / sum_s w_s, w_s = exp(lse_s - max),
// lse = max + log(sum_s w_s); no contribution gives out = 0, lse = -inf.
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const int32_t* __restrict__ block_idx,
                                                      const uint16_t* __restrict__ part_o,
                                                      const float* __restrict__ part_lse, int64_t N, int H_q, int G,
                                                      int gs, int k, int64_t nb, int64_t T0,
                                                      uint16_t* __restrict__ out, float* __restrict__ lse) {
  extern __shared__ float cw[];          // [k][H_q] weights, then [H_q] 1/L
  __shared__ uint32_t use_mask[64];      // per group: bit s set if slot s contributes
  float* inv_l = cw + k * H_q;
  const int tid = threadIdx.x;
  const int64_t tr = blockIdx.x;
  const int64_t t = T0 + tr;
  for (int g = tid; g < G; g += blockDim.x) {
    const int32_t* sel = block_idx + ((int64_t)g * N + t) * k;
    uint32_t use = 0;
    for (int s = 0; s < k; ++s) {
      int32_t b = sel[s];
      bool ok = b >= 0 && (int64_t)b < nb;
      for (int s2 = 0; s2 < s && ok; ++s2) ok = sel[s2] != b;
      use |= (ok ? 1u : 0u) << s;
    }
    use_mask[g] = use;
  }
  __syncthreads();
  const float* pl = part_lse + tr * k * H_q;
  for (int i = tid; i < k * H_q; i += blockDim.x) {
    const int s = i / H_q, h = i % H_q;
    cw[i] = (use_mask[h / gs] >> s & 1u) ? pl[i] : __int_as_float(0xff800000);
  }
  __syncthreads();
  for (int h = tid; h < H_q; h += blockDim.x) {
    float m = __int_as_float(0xff800000);
    for (int s = 0; s < k; ++s) m = fmaxf(m, cw[s * H_q + h]);
    float L = 0.f;
    if (m != __int_as_float(0xff800000)) {
      for (int s = 0; s < k; ++s) {
        float w = __expf(cw[s * H_q + h] - m);  // exp(-inf) = 0 for unused slots
        cw[s * H_q + h] = w;
        L += w;
      }
    } else {
      for (int s = 0; s < k; ++s) cw[s * H_q + h] = 0.f;
    }
    inv_l[h] = L > 0.f ? 1.f / L : 0.f;
    lse[(int64_t)h * N + t] = L > 0.f ? m + logf(L) : __int_as_float(0xff800000);
  }
  __syncthreads();
  constexpr int C8 = D / 8;
  const uint16_t* po = part_o + tr * k * H_q * D;
  for (int i = tid; i < H_q * C8; i += blockDim.x) {
    const int h = i / C8, c8 = i % C8;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll 4
    for (int s = 0; s < k; ++s) {
      const float w = cw[s * H_q + h];
      if (w == 0.f) continue;
      const uint4 v = *reinterpret_cast<const uint4*>(po + ((int64_t)s * H_q + h) * D + c8 * 8);
      acc[0] = fmaf(w, bf16_lo(v.x), acc[0]);
      acc[1] = fmaf(w, bf16_hi(v.x), acc[1]);
      acc[2] = fmaf(w, bf16_lo(v.y), acc[2]);
      acc[3] = fmaf(w, bf16_hi(v.y), acc[3]);
      acc[4] = fmaf(w, bf16_lo(v.z), acc[4]);
      acc[5] = fmaf(w, bf16_hi(v.z), acc[5]);
      acc[6] = fmaf(w, bf16_lo(v.w), acc[6]);
      acc[7] = fmaf(w, bf16_hi(v.w), acc[7]);
    }
    const float il = inv_l[h];
    uint4 o;
    o.x = pack_bf16x2(acc[0] * il, acc[1] * il);
    o.y = pack_bf16x2(acc[2] * il, acc[3] * il);
    o.z = pack_bf16x2(acc[4] * il, acc[5] * il);
    o.w = pack_bf16x2(acc[6] * il, acc[7] * il);
    *reinterpret_cast<uint4*>(out + (t * H_q + h) * D + c8 * 8) = o;
  }
}

// ---------------------------------------------------------------- scratch layout
struct AttnScratch {
  int32_t *row_ptr, *entries, *n_entries;
  InvertScratch inv;
  int32_t *lo, *cnt, *tiles, *tile_off;
  uint16_t* part_o;
  float* part_lse;
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
  s.part_o = (uint16_t*)take((size_t)p.slab * p.k * p.H_q * p.d * 2);
  s.part_lse = (float*)take((size_t)p.slab * p.k * p.H_q * 4);
  if (out) *out = s;
  return off;
}

template <int D, int BK>
cudaError_t launch_tiles(const void* q, const void* k, const void* v, const AttnScratch& sc, const AttnPlan& p,
                         int64_t T0, float scale, cudaStream_t s) {
  constexpr int LDS = D + 8;
  const size_t smem = (size_t)(kTileRows + 2 * BK) * LDS * 2;
  auto kern = attn_tile_kernel<D, BK>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = num_sms() * 2;
  kern<<<grid, kAttnThreads, smem, s>>>((const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)v, sc.entries,
                                        sc.lo, sc.cnt, sc.tile_off, p.N, p.H_q, p.H_kv, p.k, p.nb, p.gs, p.P, T0,
                                        scale * 1.4426950408889634f, sc.part_o, sc.part_lse);
  return cudaGetLastError();
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
  p.P = kTileRows / p.gs;
  // partial results of one slab: slab * k * H_q * (2d + 4) bytes, at most ~36 GB
  const double per_pos = (double)k * H_q * (2.0 * d + 4.0);
  int64_t cap = (int64_t)(36.0e9 / per_pos);
  if (cap > 131072) cap = 131072;
  if (cap < 1024) cap = 1024;
  p.slab = N < cap ? N : cap;
  return p;
}

size_t attn_scratch_bytes(const AttnPlan& p) { return carve(p, nullptr, nullptr); }

cudaError_t launch_attn(const void* q, const void* k, const void* v, const int32_t* block_idx, const AttnPlan& p,
                        float scale, void* out, float* lse, void* scratch, DeviceStatus* st, cudaStream_t s) {
  AttnScratch sc;
  carve(p, scratch, &sc);
  const int G = p.H_kv;
  cudaError_t e = launch_invert(block_idx, p.N, G, p.Bk, p.k, sc.row_ptr, sc.entries, sc.n_entries, sc.inv, st, s);
  if (e != cudaSuccess) return e;
  const int64_t n_gb = (int64_t)G * p.nb;
  for (int64_t T0 = 0; T0 < p.N; T0 += p.slab) {
    const int64_t T1 = T0 + p.slab < p.N ? T0 + p.slab : p.N;
    sched_count_kernel<<<(unsigned)((n_gb + 255) / 256), 256, 0, s>>>(sc.row_ptr, sc.entries, p.N, G, p.k, p.nb, T0,
                                                                      T1, p.P, sc.lo, sc.cnt, sc.tiles);
    sched_scan_kernel<<<1, 1024, 0, s>>>(sc.tiles, n_gb, sc.tile_off);
    if (p.d == 64 && p.Bk == 64) e = launch_tiles<64, 64>(q, k, v, sc, p, T0, scale, s);
    else if (p.d == 64) e = launch_tiles<64, 128>(q, k, v, sc, p, T0, scale, s);
    else if (p.Bk == 64) e = launch_tiles<128, 64>(q, k, v, sc, p, T0, scale, s);
    else e = launch_tiles<128, 128>(q, k, v, sc, p, T0, scale, s);
    if (e != cudaSuccess) return e;
    const size_t cs = ((size_t)p.k * p.H_q + p.H_q) * sizeof(float);
    auto ck = p.d == 64 ? combine_kernel<64> : combine_kernel<128>;
    if (cs > 48 * 1024) {
      e = cudaFuncSetAttribute(ck, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cs);
      if (e != cudaSuccess) return e;
    }
    ck<<<(unsigned)(T1 - T0), 256, cs, s>>>(block_idx, sc.part_o, sc.part_lse, p.N, p.H_q, G, p.gs, p.k, p.nb, T0,
                                            (uint16_t*)out, lse);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace msa
