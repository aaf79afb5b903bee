// msa_decode: one decode step for B sequences.
//
// velog llama.cpp analysis, section 2 (each step scans the whole 256 B/token
// index-key cache; the K/V read is fixed at the selected blocks) and section 4
// (block scores -> max-pooling -> forced local block + top-k -> attention over
// the selected blocks); "MSA" study note 2-3 for the equations.
//
//   1. scan:    split-K over the cache.  Each warp streams 16 index keys at a
//               time straight from HBM into MMA A-fragments (16-byte loads,
//               dims permuted consistently in the query fragments, so no
//               shared-memory staging is needed) and scores all groups at once
//               (16 keys x 8 groups x d_I per mma chain); block maxima feed a
//               per-group top-(k-1) list per warp, merged per CTA.
//   2. merge:   per (sequence, group) a tournament over the CTAs' candidate
//               lists -> block set.
//   3. attend:  per (sequence, group, slot) one CTA reads that block's K/V
//               rows and produces each group head's partial (O, lse).
//   4. combine: per (sequence, head) the partials are merged by their lse.
#include <math.h>

#include <mutex>

#include "msa_sm100.cuh"

namespace msa {

namespace {

constexpr int kScanThreads = 256;  // 8 warps
constexpr int kGroupsPerMma = 8;   // mma n = 8 groups

// dims of fragment column kf (0..15) in k-step ks: see the load pattern below
__device__ __forceinline__ int frag_dim(int ks, int kf) {
  int p = ks >> 1, half = ks & 1;
  int c = (kf & 7) >> 1, e = kf & 1, hi = kf >> 3;
  return 32 * p + 8 * c + 4 * half + 2 * hi + e;
}

template <int DI, int BK, int CAP>
__global__ void __launch_bounds__(kScanThreads) decode_scan_kernel(
    const uint16_t* __restrict__ q_idx_t, const uint16_t* __restrict__ k_idx_cache,
    const int32_t* __restrict__ ctx_len, int64_t ctx_max, int G, int k, int splits, float* __restrict__ cand_s,
    int32_t* __restrict__ cand_b, DeviceStatus* st) {
  constexpr int KS = DI / 16;
  __shared__ float sm_s[kScanThreads / 32][kGroupsPerMma][CAP];
  __shared__ int32_t sm_b[kScanThreads / 32][kGroupsPerMma][CAP];
  const int seq = blockIdx.y, split = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = lane & 3, row = lane >> 2;
  const int64_t len = ctx_len[seq];
  const bool ok = len >= 1 && len <= ctx_max;
  if (!ok && split == 0 && tid == 0) raise_error(st, kErrBadIndex, 2u);
  const int64_t t = ok ? len - 1 : 0;
  const int64_t local = t / BK;  // candidates: blocks [0, local)
  const int64_t b_lo = ok ? local * split / splits : 0, b_hi = ok ? local * (split + 1) / splits : 0;

  // query fragments (B operand): column n = group, k rows follow frag_dim
  uint32_t qf[KS][2];
  {
    const int n = row;  // group of this thread's B column
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        uint32_t w = 0;
        if (n < G) {
          const uint16_t* qp = q_idx_t + ((int64_t)seq * G + n) * DI;
          int d0 = frag_dim(ks, 2 * c + 8 * r), d1 = frag_dim(ks, 2 * c + 1 + 8 * r);
          w = (uint32_t)qp[d0] | ((uint32_t)qp[d1] << 16);
        }
        qf[ks][r] = w;
      }
  }

  TopK<CAP> top;
  top.init(lane < G ? k - 1 : 0);
  const uint16_t* cache = k_idx_cache + (int64_t)seq * ctx_max * DI;

  for (int64_t b = b_lo + warp; b < b_hi; b += kScanThreads / 32) {
    float bm0 = __int_as_float(0xff800000), bm1 = bm0;
#pragma unroll 2
    for (int it = 0; it < BK / 16; ++it) {
      const int64_t key = b * BK + it * 16 + row;
      const uint16_t* pa = cache + key * DI + 8 * c;
      const uint16_t* pb = pa + 8 * DI;
      uint4 va[DI / 32], vb[DI / 32];
#pragma unroll
      for (int p = 0; p < DI / 32; ++p) {
        va[p] = ldg_stream_16(pa + 32 * p);
        vb[p] = ldg_stream_16(pb + 32 * p);
      }
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int p = 0; p < DI / 32; ++p) {
        uint32_t a0[4] = {va[p].x, vb[p].x, va[p].y, vb[p].y};  // k-step 2p: dims +0..3 of each 8
        uint32_t a1[4] = {va[p].z, vb[p].z, va[p].w, vb[p].w};  // k-step 2p+1: dims +4..7
        mma_bf16_16816(acc, a0, qf[2 * p]);
        mma_bf16_16816(acc, a1, qf[2 * p + 1]);
      }
      bm0 = fmaxf(bm0, fmaxf(acc[0], acc[2]));  // group 2c, keys row and row+8
      bm1 = fmaxf(bm1, fmaxf(acc[1], acc[3]));  // group 2c+1
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, o));
      bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, o));
    }
    // group g's maximum sits in lane g/2 (value g&1)
    float x0 = __shfl_sync(0xffffffffu, bm0, (lane & 7) >> 1);
    float x1 = __shfl_sync(0xffffffffu, bm1, (lane & 7) >> 1);
    if (lane < G) top.insert((lane & 1) ? x1 : x0, (int)b);
  }

  // merge the warps' lists: lane g of warp 0 collects group g
  if (lane < kGroupsPerMma) {
    int32_t ids[CAP];
    float scs[CAP];
    int n = top.emit(CAP, ids, scs);
    for (int i = 0; i < CAP; ++i) {
      sm_s[warp][lane][i] = i < n ? scs[i] : __int_as_float(0xff800000);
      sm_b[warp][lane][i] = i < n ? ids[i] : -1;
    }
  }
  __syncthreads();
  if (warp == 0 && lane < G) {
    TopK<CAP> m;
    m.init(k - 1);
    for (int w = 0; w < kScanThreads / 32; ++w)
      for (int i = 0; i < CAP; ++i)
        if (sm_b[w][lane][i] >= 0) m.insert(sm_s[w][lane][i], sm_b[w][lane][i]);
    int32_t ids[CAP];
    float scs[CAP];
    int n = m.emit(CAP, ids, scs);
    const int64_t base = (((int64_t)seq * splits + split) * G + lane) * CAP;
    for (int i = 0; i < CAP; ++i) {
      cand_s[base + i] = i < n ? scs[i] : __int_as_float(0xff800000);
      cand_b[base + i] = i < n ? ids[i] : -1;
    }
  }
}

// One CTA per (sequence, group): a tournament over the scan CTAs' candidate
// lists (each sorted best-first).  Thread i holds the head of list i (and of
// lists i + blockDim, ...); each of the k-1 rounds takes the best head in the
// CTA (larger score, then smaller block id) and advances the winner's list.
template <int CAP>
__global__ void __launch_bounds__(1024) decode_merge_kernel(const float* __restrict__ cand_s,
                                                            const int32_t* __restrict__ cand_b,
                                                            const int32_t* __restrict__ ctx_len, int64_t ctx_max,
                                                            int Bk, int G, int k, int splits,
                                                            int32_t* __restrict__ block_idx) {
  __shared__ uint64_t warp_best[32];
  const int seq = blockIdx.x, g = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int64_t len = ctx_len[seq];
  int32_t* out = block_idx + ((int64_t)seq * G + g) * k;
  if (len < 1 || len > ctx_max) {
    for (int i = tid; i < k; i += blockDim.x) out[i] = -1;
    return;
  }
  // this thread's lists: tid, tid + blockDim, ...; pos[] = next unread entry of each
  auto list_base = [&](int sp) { return (((int64_t)seq * splits + sp) * G + g) * CAP; };
  auto head_key = [&](int sp, int p) -> uint64_t {
    if (p >= CAP) return 0;
    const int32_t b = cand_b[list_base(sp) + p];
    return b < 0 ? 0 : rank_key(cand_s[list_base(sp) + p], b);
  };
  constexpr int kMaxLists = 4;  // lists per thread (splits <= 4 * 1024)
  int pos[kMaxLists];
  uint64_t key[kMaxLists];
#pragma unroll
  for (int i = 0; i < kMaxLists; ++i) {
    const int sp = tid + i * blockDim.x;
    pos[i] = 0;
    key[i] = sp < splits ? head_key(sp, 0) : 0;
  }
  if (tid == 0) out[0] = (int32_t)((len - 1) / Bk);
  for (int r = 0; r < k - 1; ++r) {
    uint64_t best = 0;
#pragma unroll
    for (int i = 0; i < kMaxLists; ++i) best = key[i] > best ? key[i] : best;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const uint64_t other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    if (lane == 0) warp_best[warp] = best;
    __syncthreads();
    uint64_t all = 0;
    for (int w = 0; w < nwarps; ++w) all = warp_best[w] > all ? warp_best[w] : all;
    __syncthreads();  // warp_best is rewritten next round
    if (tid == 0) out[1 + r] = all == 0 ? -1 : (int32_t)(0xFFFFFFFFu - (uint32_t)(all & 0xFFFFFFFFu));
    if (all == 0) continue;
#pragma unroll
    for (int i = 0; i < kMaxLists; ++i)
      if (key[i] == all) {  // keys are unique: block ids differ across lists
        const int sp = tid + i * blockDim.x;
        key[i] = head_key(sp, ++pos[i]);
      }
  }
}

// One CTA per (slot, group, sequence): 128 threads.
// One CTA (4 warps) per (slot, group, sequence): the block's K/V rows are
// staged in shared memory (16-byte chunk c of row j stored at chunk
// c ^ (j mod d/8), so ldmatrix rows fall in distinct banks).  The group's
// heads are the rows of m16n8k16 tensor-core tiles (rows >= gs are zero):
// warp w scores keys [w BK/4, (w+1) BK/4), the softmax statistics are merged
// across warps in shared memory, P stays in registers as the A operand of
// P V (V read transposed by ldmatrix), and the warps' partial O are summed in
// shared memory before the head's partial (O, lse) is written.
template <int D, int BK>
__global__ void __launch_bounds__(128) decode_attn_kernel(const uint16_t* __restrict__ q_t,
                                                          const uint16_t* __restrict__ k_cache,
                                                          const uint16_t* __restrict__ v_cache,
                                                          const int32_t* __restrict__ ctx_len,
                                                          const int32_t* __restrict__ block_idx, int64_t ctx_max,
                                                          int H_q, int G, int k, float scale,
                                                          float* __restrict__ part_o, float* __restrict__ part_lse) {
  extern __shared__ __align__(16) uint16_t kv_s[];  // K rows [BK][D], then V rows [BK][D]
  __shared__ float red_m[4][8], red_l[4][8];
  constexpr int C8 = D / 8;     // 16-byte chunks per row
  constexpr int KPW = BK / 4;   // keys per warp
  constexpr int NT = KPW / 8;   // 8-key n-tiles per warp
  constexpr int KS = D / 16;    // k-steps over d
  static_assert(NT % 2 == 0, "two n-tiles per ldmatrix");
  const int slot = blockIdx.x, g = blockIdx.y, seq = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;  // fragment row (head) and column pair
  const int gs = H_q / G;
  const int64_t len = ctx_len[seq];
  const int32_t b = block_idx[((int64_t)seq * G + g) * k + slot];
  const int64_t nb = (ctx_max + BK - 1) / BK;
  const bool valid = len >= 1 && len <= ctx_max && b >= 0 && (int64_t)b < nb;
  const int64_t t = len - 1;
  const int64_t key0 = (int64_t)b * BK;
  const int nvis = valid ? (int)max((int64_t)0, min((int64_t)BK, t - key0 + 1)) : 0;
  float* po = part_o + (((int64_t)seq * H_q + g * gs) * k + slot) * D;
  float* pl = part_lse + ((int64_t)seq * H_q + g * gs) * k + slot;
  if (nvis == 0) {
    for (int hh = tid; hh < gs; hh += blockDim.x) pl[(int64_t)hh * k] = __int_as_float(0xff800000);
    return;
  }
  // stage the visible K and V rows with every copy in flight at once (rows past nvis read as zero)
  const int64_t kv_row = (int64_t)G * D;
  const uint16_t* Kb = k_cache + ((int64_t)seq * ctx_max + key0) * kv_row + (int64_t)g * D;
  const uint16_t* Vb = v_cache + ((int64_t)seq * ctx_max + key0) * kv_row + (int64_t)g * D;
  uint16_t* Ks = kv_s;
  uint16_t* Vs = kv_s + BK * D;
  for (int i = tid; i < BK * C8; i += blockDim.x) {
    const int j = i / C8, c8 = i % C8;
    const bool in = j < nvis;
    const int64_t off = (int64_t)(in ? j : 0) * kv_row + c8 * 8;
    const int sw = (c8 ^ (j & (C8 - 1))) * 8;
    cp_async_16(Ks + j * D + sw, Kb + off, in ? 16 : 0);
    cp_async_16(Vs + j * D + sw, Vb + off, in ? 16 : 0);
  }
  cp_async_commit();
  // q as A fragments: row gq = head gq of the group (zero past gs), rows 8..15 zero
  uint32_t qa[KS][2];
  {
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(q_t + ((int64_t)seq * H_q + g * gs + gq) * D);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][0] = gq < gs ? qrow[(16 * ks + 2 * tq) >> 1] : 0u;
      qa[ks][1] = gq < gs ? qrow[(16 * ks + 8 + 2 * tq) >> 1] : 0u;
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  // S = q K^T for this warp's keys
  float sacc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const uint32_t a[4] = {qa[ks][0], 0u, qa[ks][1], 0u};
#pragma unroll
    for (int np = 0; np < NT; np += 2) {
      // matrices: (n-tile np, dims +0..7), (np, +8..15), (np+1, +0..7), (np+1, +8..15)
      const int key = warp * KPW + np * 8 + (lane & 7) + ((lane >> 4) << 3);
      const int chunk = 2 * ks + ((lane >> 3) & 1);
      uint32_t r0, r1, r2, r3;
      ldmatrix_x4(r0, r1, r2, r3, Ks + key * D + ((chunk ^ (key & (C8 - 1))) * 8));
      const uint32_t b0[2] = {r0, r1}, b1[2] = {r2, r3};
      mma_bf16_16816(sacc[np], a, b0);
      mma_bf16_16816(sacc[np + 1], a, b1);
    }
  }
  // scale, mask past nvis, row (head) maxima across the warp's keys and then across warps
  float mx = __int_as_float(0xff800000);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int j = warp * KPW + nt * 8 + 2 * tq + e;
      const float v = j < nvis ? sacc[nt][e] * scale : __int_as_float(0xff800000);
      sacc[nt][e] = v;
      mx = fmaxf(mx, v);
    }
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  if (tq == 0) red_m[warp][gq] = mx;
  __syncthreads();
  const float m = fmaxf(fmaxf(red_m[0][gq], red_m[1][gq]), fmaxf(red_m[2][gq], red_m[3][gq]));
  float ls = 0.f;
  uint32_t pa[NT / 2][2];  // P as A fragments of the P V k-steps (16 keys each)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float p0 = __expf(sacc[nt][0] - m), p1 = __expf(sacc[nt][1] - m);  // e^-inf = 0
    ls += p0 + p1;
    pa[nt >> 1][nt & 1] = pack_bf16x2(p0, p1);
  }
  ls += __shfl_xor_sync(0xffffffffu, ls, 1);
  ls += __shfl_xor_sync(0xffffffffu, ls, 2);
  if (tq == 0) red_l[warp][gq] = ls;
  // O = P V over this warp's keys
  float oacc[D / 8][4];
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd) oacc[nd][0] = oacc[nd][1] = oacc[nd][2] = oacc[nd][3] = 0.f;
#pragma unroll
  for (int ks2 = 0; ks2 < NT / 2; ++ks2) {
    const uint32_t a[4] = {pa[ks2][0], 0u, pa[ks2][1], 0u};
#pragma unroll
    for (int nd = 0; nd < D / 8; nd += 2) {
      // transposed matrices: (keys +0..7, d n-tile nd), (keys +8..15, nd), (+0..7, nd+1), (+8..15, nd+1)
      const int key = warp * KPW + 16 * ks2 + (lane & 7) + (((lane >> 3) & 1) << 3);
      const int chunk = nd + (lane >> 4);
      uint32_t r0, r1, r2, r3;
      ldmatrix_x4_trans(r0, r1, r2, r3, Vs + key * D + ((chunk ^ (key & (C8 - 1))) * 8));
      const uint32_t b0[2] = {r0, r1}, b1[2] = {r2, r3};
      mma_bf16_16816(oacc[nd], a, b0);
      mma_bf16_16816(oacc[nd + 1], a, b1);
    }
  }
  // sum the warps' partial O in shared memory (over the K rows, which are no longer read)
  __syncthreads();
  float* red_o = reinterpret_cast<float*>(kv_s);  // [4 warps][8 rows][D]
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd) {
    red_o[(warp * 8 + gq) * D + nd * 8 + 2 * tq] = oacc[nd][0];
    red_o[(warp * 8 + gq) * D + nd * 8 + 2 * tq + 1] = oacc[nd][1];
  }
  __syncthreads();
  for (int i = tid; i < gs * D; i += blockDim.x) {
    const int hh = i / D, dc = i % D;
    const float L = red_l[0][hh] + red_l[1][hh] + red_l[2][hh] + red_l[3][hh];
    const float o = red_o[(0 * 8 + hh) * D + dc] + red_o[(1 * 8 + hh) * D + dc] + red_o[(2 * 8 + hh) * D + dc] +
                    red_o[(3 * 8 + hh) * D + dc];
    po[(int64_t)hh * k * D + dc] = o / L;
  }
  if (tid < gs) {
    const float M = fmaxf(fmaxf(red_m[0][tid], red_m[1][tid]), fmaxf(red_m[2][tid], red_m[3][tid]));
    const float L = red_l[0][tid] + red_l[1][tid] + red_l[2][tid] + red_l[3][tid];
    pl[(int64_t)tid * k] = M + logf(L);
  }
}

template <int D>
__global__ void decode_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse, int H_q,
                                      int k, uint16_t* __restrict__ out, float* __restrict__ lse) {
  const int64_t sh = blockIdx.x;  // seq * H_q + h
  const float* pl = part_lse + sh * k;
  float m = __int_as_float(0xff800000);
  for (int s = 0; s < k; ++s) m = fmaxf(m, pl[s]);
  for (int cc = threadIdx.x; cc < D; cc += blockDim.x) {
    float acc = 0.f, L = 0.f;
    if (m != __int_as_float(0xff800000)) {
      for (int s = 0; s < k; ++s) {
        if (pl[s] == __int_as_float(0xff800000)) continue;
        float w = __expf(pl[s] - m);
        L += w;
        acc += w * part_o[(sh * k + s) * D + cc];
      }
    }
    out[sh * D + cc] = (uint16_t)(pack_bf16x2(L > 0.f ? acc / L : 0.f, 0.f) & 0xFFFFu);
    if (cc == 0 && lse) lse[sh] = L > 0.f ? m + logf(L) : __int_as_float(0xff800000);
  }
}

struct DecodeScratch {
  float* cand_s;
  int32_t* cand_b;
  int32_t* blk;
  float* part_o;
  float* part_lse;
};

static size_t carve(const DecodePlan& p, void* base, DecodeScratch* out) {
  char* c = (char*)base;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* r = c ? c + off : nullptr;
    off += align_up(bytes, 256);
    return r;
  };
  const int cap = topk_cap(p.k - 1);
  DecodeScratch s;
  s.cand_s = (float*)take((size_t)p.B * p.splits * p.H_kv * cap * 4);
  s.cand_b = (int32_t*)take((size_t)p.B * p.splits * p.H_kv * cap * 4);
  s.blk = (int32_t*)take((size_t)p.B * p.H_kv * p.k * 4);
  s.part_o = (float*)take((size_t)p.B * p.H_q * p.k * p.d * 4);
  s.part_lse = (float*)take((size_t)p.B * p.H_q * p.k * 4);
  if (out) *out = s;
  return off;
}

template <int DI, int BK, int CAP>
cudaError_t launch_scan_merge(const void* q_idx_t, const void* k_idx_cache, const int32_t* ctx_len,
                              const DecodePlan& p, const DecodeScratch& sc, int32_t* blk, DeviceStatus* st,
                              cudaStream_t s) {
  dim3 grid((unsigned)p.splits, (unsigned)p.B);
  decode_scan_kernel<DI, BK, CAP><<<grid, kScanThreads, 0, s>>>((const uint16_t*)q_idx_t,
                                                                (const uint16_t*)k_idx_cache, ctx_len, p.ctx_max,
                                                                p.H_kv, p.k, p.splits, sc.cand_s, sc.cand_b, st);
  const int mthreads = p.splits >= 1024 ? 1024 : (p.splits + 31) / 32 * 32;
  decode_merge_kernel<CAP><<<dim3((unsigned)p.B, (unsigned)p.H_kv), mthreads, 0, s>>>(
      sc.cand_s, sc.cand_b, ctx_len, p.ctx_max, p.Bk, p.H_kv, p.k, p.splits, blk);
  return cudaGetLastError();
}

template <int DI, int BK>
cudaError_t scan_cap(const void* a, const void* b, const int32_t* c, const DecodePlan& p, const DecodeScratch& sc,
                     int32_t* blk, DeviceStatus* st, cudaStream_t s) {
  int km1 = p.k - 1;
  if (km1 <= 4) return launch_scan_merge<DI, BK, 4>(a, b, c, p, sc, blk, st, s);
  if (km1 <= 8) return launch_scan_merge<DI, BK, 8>(a, b, c, p, sc, blk, st, s);
  if (km1 <= 16) return launch_scan_merge<DI, BK, 16>(a, b, c, p, sc, blk, st, s);
  return launch_scan_merge<DI, BK, 32>(a, b, c, p, sc, blk, st, s);
}

}  // namespace

DecodePlan decode_plan(int B, int64_t ctx_max, int H_q, int H_kv, int d, int d_I, int Bk, int k) {
  DecodePlan p;
  p.B = B;
  p.ctx_max = ctx_max;
  p.H_q = H_q;
  p.H_kv = H_kv;
  p.d = d;
  p.d_I = d_I;
  p.Bk = Bk;
  p.k = k;
  p.gs = H_q / H_kv;
  const int64_t nb = (ctx_max + Bk - 1) / Bk;
  int64_t splits = ((int64_t)num_sms() * 4 + B - 1) / B;  // ~4 CTAs of 8 warps per SM
  int64_t max_splits = nb / 8 > 1 ? nb / 8 : 1;             // at least 8 blocks per CTA
  if (splits > max_splits) splits = max_splits;
  if (splits < 1) splits = 1;
  p.splits = (int)splits;
  return p;
}

size_t decode_scratch_bytes(const DecodePlan& p) { return carve(p, nullptr, nullptr); }

cudaError_t launch_decode(const void* q_t, const void* q_idx_t, const void* k_idx_cache, const void* k_cache,
                          const void* v_cache, const int32_t* ctx_len, const DecodePlan& p, float scale, void* out,
                          float* lse, int32_t* block_idx, void* scratch, DeviceStatus* st, cudaStream_t s) {
  DecodeScratch sc;
  carve(p, scratch, &sc);
  int32_t* blk = block_idx ? block_idx : sc.blk;
  cudaError_t e;
  if (p.d_I == 32) {
    e = p.Bk == 64 ? scan_cap<32, 64>(q_idx_t, k_idx_cache, ctx_len, p, sc, blk, st, s)
                   : scan_cap<32, 128>(q_idx_t, k_idx_cache, ctx_len, p, sc, blk, st, s);
  } else if (p.d_I == 64) {
    e = p.Bk == 64 ? scan_cap<64, 64>(q_idx_t, k_idx_cache, ctx_len, p, sc, blk, st, s)
                   : scan_cap<64, 128>(q_idx_t, k_idx_cache, ctx_len, p, sc, blk, st, s);
  } else {
    e = p.Bk == 64 ? scan_cap<128, 64>(q_idx_t, k_idx_cache, ctx_len, p, sc, blk, st, s)
                   : scan_cap<128, 128>(q_idx_t, k_idx_cache, ctx_len, p, sc, blk, st, s);
  }
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.k, (unsigned)p.H_kv, (unsigned)p.B);
  auto attn_smem = [](int D, int BK) { return 2 * BK * D * 2; };  // K and V rows of one block
  if (p.d == 128 && p.Bk == 128) {
    e = cudaFuncSetAttribute(decode_attn_kernel<128, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             attn_smem(128, 128));
    if (e != cudaSuccess) return e;
  }
  if (p.d == 64 && p.Bk == 64)
    decode_attn_kernel<64, 64><<<grid, 128, attn_smem(64, 64), s>>>((const uint16_t*)q_t, (const uint16_t*)k_cache,
                                                    (const uint16_t*)v_cache, ctx_len, blk, p.ctx_max, p.H_q, p.H_kv,
                                                    p.k, scale, sc.part_o, sc.part_lse);
  else if (p.d == 64)
    decode_attn_kernel<64, 128><<<grid, 128, attn_smem(64, 128), s>>>((const uint16_t*)q_t, (const uint16_t*)k_cache,
                                                     (const uint16_t*)v_cache, ctx_len, blk, p.ctx_max, p.H_q,
                                                     p.H_kv, p.k, scale, sc.part_o, sc.part_lse);
  else if (p.Bk == 64)
    decode_attn_kernel<128, 64><<<grid, 128, attn_smem(128, 64), s>>>((const uint16_t*)q_t, (const uint16_t*)k_cache,
                                                     (const uint16_t*)v_cache, ctx_len, blk, p.ctx_max, p.H_q,
                                                     p.H_kv, p.k, scale, sc.part_o, sc.part_lse);
  else
    decode_attn_kernel<128, 128><<<grid, 128, attn_smem(128, 128), s>>>((const uint16_t*)q_t, (const uint16_t*)k_cache,
                                                      (const uint16_t*)v_cache, ctx_len, blk, p.ctx_max, p.H_q,
                                                      p.H_kv, p.k, scale, sc.part_o, sc.part_lse);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (p.d == 64)
    decode_combine_kernel<64><<<p.B * p.H_q, 64, 0, s>>>(sc.part_o, sc.part_lse, p.H_q, p.k, (uint16_t*)out, lse);
  else
    decode_combine_kernel<128><<<p.B * p.H_q, 128, 0, s>>>(sc.part_o, sc.part_lse, p.H_q, p.k, (uint16_t*)out, lse);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- fixed scratch for msa_decode_noalloc
// Scratch of the decode step for callers that cannot allocate device memory:
// a file-scope device array, resident on every GPU that loads the library
// until the process exits.  In host code `g_noalloc_scratch` names a host-side
// shadow, not device memory, so kernels only ever receive the address looked
// up below with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

cudaError_t noalloc_scratch(size_t need, void** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  *out = nullptr;
  if (need > kNoAllocScratchBytes) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {  // once per device, with that device current
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace msa
