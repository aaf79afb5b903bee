// Warmup mode: dense main attention and the index branch's full-context KL.
//
// "MSA" study note 4-4 "Indexer warmup": before top-k routing is switched on,
// the main branch runs full attention and the index branch learns the KL
// alignment against the full-context teacher (4-2: the teacher is the mean of
// the GQA group's main-branch probabilities; 4-3: it is detached and the KL
// reaches only q^I and k^I); 1-1 for dense causal GQA attention.
//
// Per row (t, h), g = h / gs, over every key j <= t:
//   z = scale q.k_j, out = softmax(z) V, lse = logsumexp(z);
// per row (t, g): pbar_j = mean_h exp(z_{h,j} - lse_h), zI_j = q^I.k^I_j /
// sqrt(d_I), lse^I = logsumexp(zI), KL = sum_j pbar_j (log pbar_j - zI_j +
// lse^I), dzI_j = w (exp(zI_j - lse^I) - pbar_j),
//   dq^I = sum_j dzI_j k^I_j / sqrt(d_I), dk^I_j += dzI_j q^I / sqrt(d_I).
//
// Three mma.sync kernels over tiles of 16 positions x 8 head slots (128 rows,
// slots >= gs are zero rows) and 64-key tiles, 8 warps (warp w owns rows
// 16w..16w+15, i.e. positions 2w and 2w+1):
//   fwd:    query-outer; online softmax and P V per warp, and the index
//           logits of the 16 positions (warps 0-3, 16 keys each) with a
//           per-thread online logsumexp -> out, lse, lse^I;
//   dq:     query-outer; per key tile the dz tile (below), KL per row, and
//           dq^I += dz K^I (warp w: 16 of the d_I columns);
//   dk:     key-outer (one 64-key tile per CTA); per query tile the dz tile
//           and dk^I += dz^T Q^I, flushed once with fp32 reductions over the
//           groups.
// The dz tile: S recomputed for the 128 rows, P = exp(scale S - lse), the
// teacher summed over each position's 8 rows by a shuffle reduce-scatter (each
// lane ends with 4 of the warp's 32 x 2 teacher entries), the index logits
// through shared memory, dz (bf16) into shared memory.  K/V (or Q) tiles are
// double-buffered with cp.async.
#include <math.h>

#include "msa_common.cuh"
#include "msa_internal.h"
#include "msa_tiles.cuh"

namespace msa {

namespace {

using namespace tiles;

constexpr int kWPos = 16;     // positions per query tile
constexpr int kWRows = 128;   // 16 positions x 8 head slots
constexpr int kWKeys = 64;    // keys per key tile
constexpr int kWThreads = 256;
constexpr float kNegInf = -INFINITY;

template <int D, int DI>
struct WarmSmem {
  static constexpr int Q = kWRows * D * 2;     // one query tile (128 rows)
  static constexpr int QI = kWPos * DI * 2;    // its index queries
  static constexpr int K = kWKeys * D * 2;     // one key tile
  static constexpr int KI = kWKeys * DI * 2;   // its index keys
  static constexpr int ZI = kWPos * kWKeys * 4;  // index logits of a tile (fp32)
  static constexpr int DZ = kWPos * kWKeys * 2;  // dz of a tile (bf16)
};

// Rows of a query tile: row r = position (r >> 3), head slot (r & 7).
__device__ __forceinline__ const uint16_t* q_row(const uint16_t* q, int64_t t0, int r, int64_t N, int H_q, int g,
                                                 int gs, int D) {
  const int64_t t = t0 + (r >> 3);
  const int hh = r & 7;
  return (t < N && hh < gs) ? q + (t * H_q + (int64_t)g * gs + hh) * D : nullptr;
}

// ------------------------------------------------------------------ the dz tile
// Query tile [t0, t0+16) (rows in Qs, index queries in qIs) against key tile
// [j0, j0+64) (Ks, kIs), for the warp's rows; lse_r[2]: the main lse of its
// rows gq, gq+8 (-inf for padding rows); lseI_p[2]: lse^I of its positions
// 2w, 2w+1.  Writes dz (bf16) of the 16 positions x 64 keys into dz_s and, with
// KL, adds the KL terms of its positions to kl_acc (spread over the warp's lanes).
template <int D, int DI, bool KL>
__device__ __forceinline__ void dz_tile(uint32_t Qs, uint32_t qIs, uint32_t Ks, uint32_t kIs, float* zI_s,
                                        uint16_t* dz_s, int64_t t0, int64_t j0, int64_t N, float scale, float sI,
                                        float w_kl, const float (&lse_r)[2], const float (&lseI_p)[2], int gs,
                                        float (&kl_acc)[2]) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  // index logits of the 16 positions: warps 0-3, 16 keys each, into zI_s
  if (warp < 4) {
    float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < DI / 16; ++ks) {
      uint32_t a[4], b[4];
      lds_a(a, qIs, 0, 16 * ks, DI);
      lds_b_nk(b, kIs, 16 * warp, 16 * ks, DI);
      mma2(c[0], c[1], a, b);
    }
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int p = gq + ((e >> 1) << 3), col = 16 * warp + 8 * n + 2 * tq + (e & 1);
        zI_s[p * kWKeys + col] = c[n][e] * sI;
      }
  }
  // S for the warp's 16 rows x 64 keys
  float s[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    uint32_t a[4];
    lds_a(a, Qs, 16 * warp, 16 * ks, D);
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      uint32_t b[4];
      lds_b_nk(b, Ks, 16 * np, 16 * ks, D);
      mma2(s[2 * np], s[2 * np + 1], a, b);
    }
  }
  // P for the warp's rows: gq (position 2w) and gq + 8 (position 2w + 1), slot gq
  const int64_t tp[2] = {t0 + 2 * warp, t0 + 2 * warp + 1};
  float v[32];  // v[4n + e]: n-tile n, accumulator element e
#pragma unroll
  for (int n = 0; n < 8; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int ri = e >> 1;
      const int64_t j = j0 + 8 * n + 2 * tq + (e & 1);
      const bool ok = tp[ri] < N && j <= tp[ri] && gq < gs;
      v[4 * n + e] = ok ? __expf(fmaf(s[n][e], scale, -lse_r[ri])) : 0.f;
    }
  // The teacher sums each position's 8 slot rows, which sit in the 8 lanes of a
  // tq column (lane bits 2-4).  A reduce-scatter over those bits (exchange half,
  // keep half, three times) leaves lane gq with the full sums of n-tile
  // nf = 4 (gq & 1) + 2 ((gq >> 1) & 1) + (gq >> 2), elements 0..3.
  const int b0 = gq & 1, b1 = (gq >> 1) & 1, b2 = gq >> 2;
  float r1[16], r2[8], pb[4];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float keep = b0 ? v[16 + i] : v[i], send = b0 ? v[i] : v[16 + i];
    r1[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float keep = b1 ? r1[8 + i] : r1[i], send = b1 ? r1[i] : r1[8 + i];
    r2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  const float inv_gs = 1.f / (float)gs;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float keep = b2 ? r2[4 + i] : r2[i], send = b2 ? r2[i] : r2[4 + i];
    pb[i] = (keep + __shfl_xor_sync(0xffffffffu, send, 16)) * inv_gs;
  }
  const int nf = 4 * b0 + 2 * b1 + b2;
  __syncthreads();  // zI_s complete
  // dz and KL of the lane's 4 teacher entries
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int ri = e >> 1, p = 2 * warp + ri, col = 8 * nf + 2 * tq + (e & 1);
    const int64_t j = j0 + col;
    const bool ok = tp[ri] < N && j <= tp[ri];
    float dz = 0.f;
    if (ok) {
      const float lp = zI_s[p * kWKeys + col] - lseI_p[ri];  // log pI
      dz = w_kl * (__expf(lp) - pb[e]);
      if (KL && pb[e] > 0.f) kl_acc[ri] += pb[e] * (__logf(pb[e]) - lp);
    }
    st_bf16(dz_s, p, col, kWKeys, dz);
  }
  __syncthreads();  // dz_s complete
}

// ------------------------------------------------------------------ fwd
template <int D, int DI>
__global__ void __launch_bounds__(kWThreads, 1)
    warmup_fwd_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                      const uint16_t* __restrict__ v, const uint16_t* __restrict__ q_idx,
                      const uint16_t* __restrict__ k_idx, int64_t N, int H_q, int H_kv, float scale,
                      uint16_t* __restrict__ out, float* __restrict__ lse, float* __restrict__ lseI) {
  using L = WarmSmem<D, DI>;
  extern __shared__ __align__(128) uint8_t wsm[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(wsm);
  uint16_t* qIs = reinterpret_cast<uint16_t*>(wsm + L::Q);
  uint16_t* Kb = reinterpret_cast<uint16_t*>(wsm + L::Q + L::QI);               // [2][K]
  uint16_t* Vb = reinterpret_cast<uint16_t*>(wsm + L::Q + L::QI + 2 * L::K);   // [2][K]
  uint16_t* kIb = reinterpret_cast<uint16_t*>(wsm + L::Q + L::QI + 4 * L::K);  // [2][KI]
  __shared__ float red_m[4][kWPos], red_l[4][kWPos];
  const int G = H_kv, gs = H_q / H_kv;
  const int64_t n_qt = (N + kWPos - 1) / kWPos;
  const int64_t qt = n_qt - 1 - (int64_t)blockIdx.x;  // longest rows first
  const int g = blockIdx.y;
  const int64_t t0 = qt * kWPos;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const int64_t kend = min(N, t0 + kWPos);  // keys [0, kend)
  const int n_kt = (int)((kend + kWKeys - 1) / kWKeys);
  const uint16_t* kv_row = k;  // any valid address for zero-filled copies
  load_rows(Qs, kWRows, D, q, [&](int r) { return q_row(q, t0, r, N, H_q, g, gs, D); });
  load_rows(qIs, kWPos, DI, q_idx, [&](int r) {
    return t0 + r < N ? q_idx + ((t0 + r) * G + g) * DI : (const uint16_t*)nullptr;
  });
  auto load_kt = [&](int kt, int buf) {
    const int64_t j0 = (int64_t)kt * kWKeys;
    load_rows(Kb + buf * (L::K / 2), kWKeys, D, kv_row, [&](int r) {
      return j0 + r < N ? k + ((j0 + r) * H_kv + g) * D : (const uint16_t*)nullptr;
    });
    load_rows(Vb + buf * (L::K / 2), kWKeys, D, kv_row, [&](int r) {
      return j0 + r < N ? v + ((j0 + r) * H_kv + g) * D : (const uint16_t*)nullptr;
    });
    load_rows(kIb + buf * (L::KI / 2), kWKeys, DI, kv_row, [&](int r) {
      return j0 + r < N ? k_idx + (j0 + r) * DI : (const uint16_t*)nullptr;
    });
  };
  load_kt(0, 0);
  cp_async_commit();
  const int64_t tp[2] = {t0 + 2 * warp, t0 + 2 * warp + 1};
  const bool row_ok[2] = {tp[0] < N && gq < gs, tp[1] < N && gq < gs};
  float m[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f};
  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  // index: rows = positions gq and gq + 8 (warps 0-3), per-thread online logsumexp
  float mI[2] = {kNegInf, kNegInf}, lI[2] = {0.f, 0.f};
  const float sI = rsqrtf((float)DI);
  const uint32_t qs_a = smem_u32(Qs), qis_a = smem_u32(qIs);
  for (int kt = 0; kt < n_kt; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < n_kt) {
      load_kt(kt + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t ks_a = smem_u32(Kb + buf * (L::K / 2)), vs_a = smem_u32(Vb + buf * (L::K / 2));
    const uint32_t kis_a = smem_u32(kIb + buf * (L::KI / 2));
    const int64_t j0 = (int64_t)kt * kWKeys;
    // S = Q K^T (16 rows x 64 keys)
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a[4];
      lds_a(a, qs_a, 16 * warp, 16 * ks, D);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b[4];
        lds_b_nk(b, ks_a, 16 * np, 16 * ks, D);
        mma2(s[2 * np], s[2 * np + 1], a, b);
      }
    }
    // online softmax per row
    float mx[2] = {kNegInf, kNegInf};
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ri = e >> 1;
        const int64_t j = j0 + 8 * n + 2 * tq + (e & 1);
        const float x = (row_ok[ri] && j <= tp[ri]) ? s[n][e] * scale : kNegInf;
        s[n][e] = x;
        mx[ri] = fmaxf(mx[ri], x);
      }
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 1));
      mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 2));
    }
    float alpha[2];
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      const float mn = fmaxf(m[ri], mx[ri]);
      alpha[ri] = mn == kNegInf ? 1.f : __expf(m[ri] - mn);  // e^-inf = 0 on the first keys
      m[ri] = mn;
      l[ri] *= alpha[ri];
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= alpha[0];
      o[n][1] *= alpha[0];
      o[n][2] *= alpha[1];
      o[n][3] *= alpha[1];
    }
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ri = e >> 1;
        const float p = m[ri] == kNegInf ? 0.f : __expf(s[n][e] - m[ri]);
        s[n][e] = p;
        l[ri] += p;
      }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      c_to_a(pa, s[2 * kk], s[2 * kk + 1]);
#pragma unroll
      for (int nd = 0; nd < D / 16; ++nd) {
        uint32_t b[4];
        lds_b_kn(b, vs_a, 16 * kk, 16 * nd, D);
        mma2(o[2 * nd], o[2 * nd + 1], pa, b);
      }
    }
    // index logits of the 16 positions against this warp's 16 keys
    if (warp < 4) {
      float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < DI / 16; ++ks) {
        uint32_t a[4], b[4];
        lds_a(a, qis_a, 0, 16 * ks, DI);
        lds_b_nk(b, kis_a, 16 * warp, 16 * ks, DI);
        mma2(c[0], c[1], a, b);
      }
#pragma unroll
      for (int ri = 0; ri < 2; ++ri) {
        const int64_t t = t0 + gq + 8 * ri;
        float xm = kNegInf;
        float xv[4];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int64_t j = j0 + 16 * warp + 8 * n + 2 * tq + e2;
            const float x = (t < N && j <= t) ? c[n][2 * ri + e2] * sI : kNegInf;
            xv[2 * n + e2] = x;
            xm = fmaxf(xm, x);
          }
        const float mn = fmaxf(mI[ri], xm);
        if (mn != kNegInf) {
          float acc = lI[ri] * __expf(mI[ri] - mn);
#pragma unroll
          for (int i = 0; i < 4; ++i) acc += __expf(xv[i] - mn);
          lI[ri] = acc;
          mI[ri] = mn;
        }
      }
    }
    __syncthreads();  // the buffers of this tile are free for the tile after next
  }
  // main outputs
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    l[ri] += __shfl_xor_sync(0xffffffffu, l[ri], 1);
    l[ri] += __shfl_xor_sync(0xffffffffu, l[ri], 2);
  }
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    if (!row_ok[ri]) continue;
    const int h = g * gs + gq;
    const float inv = l[ri] > 0.f ? 1.f / l[ri] : 0.f;
    uint16_t* orow = out + (tp[ri] * H_q + h) * D;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      const uint32_t pk = pack_bf16x2(o[n][2 * ri] * inv, o[n][2 * ri + 1] * inv);
      *reinterpret_cast<uint32_t*>(orow + 8 * n + 2 * tq) = pk;
    }
    if (tq == 0) lse[(int64_t)h * N + tp[ri]] = m[ri] + __logf(l[ri]);
  }
  // index lse: threads -> lanes (over tq) -> warps 0-3 (through shared memory)
  if (warp < 4) {
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
#pragma unroll
      for (int o2 = 1; o2 <= 2; o2 <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, mI[ri], o2), l2 = __shfl_xor_sync(0xffffffffu, lI[ri], o2);
        const float mn = fmaxf(mI[ri], m2);
        if (mn != kNegInf) {
          lI[ri] = lI[ri] * __expf(mI[ri] - mn) + l2 * __expf(m2 - mn);
          mI[ri] = mn;
        }
      }
      if (tq == 0) {
        red_m[warp][gq + 8 * ri] = mI[ri];
        red_l[warp][gq + 8 * ri] = lI[ri];
      }
    }
  }
  __syncthreads();
  if (tid < kWPos && t0 + tid < N) {
    float M = kNegInf;
    for (int w = 0; w < 4; ++w) M = fmaxf(M, red_m[w][tid]);
    float S = 0.f;
    for (int w = 0; w < 4; ++w) S += red_m[w][tid] == kNegInf ? 0.f : red_l[w][tid] * __expf(red_m[w][tid] - M);
    lseI[(int64_t)g * N + t0 + tid] = M + __logf(S);
  }
}

// ------------------------------------------------------------------ dq (and KL)
template <int D, int DI>
__global__ void __launch_bounds__(kWThreads, 1)
    warmup_dq_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                     const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ k_idx,
                     const float* __restrict__ lse, const float* __restrict__ lseI, int64_t N, int H_q, int H_kv,
                     float scale, float w_kl, float* __restrict__ dq_idx, float* __restrict__ kl) {
  using L = WarmSmem<D, DI>;
  extern __shared__ __align__(128) uint8_t wsm[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(wsm);
  uint16_t* qIs = reinterpret_cast<uint16_t*>(wsm + L::Q);
  uint16_t* Kb = reinterpret_cast<uint16_t*>(wsm + L::Q + L::QI);               // [2][K]
  uint16_t* kIb = reinterpret_cast<uint16_t*>(wsm + L::Q + L::QI + 2 * L::K);  // [2][KI]
  float* zI_s = reinterpret_cast<float*>(wsm + L::Q + L::QI + 2 * L::K + 2 * L::KI);
  uint16_t* dz_s = reinterpret_cast<uint16_t*>(wsm + L::Q + L::QI + 2 * L::K + 2 * L::KI + L::ZI);
  const int G = H_kv, gs = H_q / H_kv;
  const int64_t n_qt = (N + kWPos - 1) / kWPos;
  const int64_t qt = n_qt - 1 - (int64_t)blockIdx.x;
  const int g = blockIdx.y;
  const int64_t t0 = qt * kWPos;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const int64_t kend = min(N, t0 + kWPos);
  const int n_kt = (int)((kend + kWKeys - 1) / kWKeys);
  load_rows(Qs, kWRows, D, q, [&](int r) { return q_row(q, t0, r, N, H_q, g, gs, D); });
  load_rows(qIs, kWPos, DI, q_idx, [&](int r) {
    return t0 + r < N ? q_idx + ((t0 + r) * G + g) * DI : (const uint16_t*)nullptr;
  });
  auto load_kt = [&](int kt, int buf) {
    const int64_t j0 = (int64_t)kt * kWKeys;
    load_rows(Kb + buf * (L::K / 2), kWKeys, D, k, [&](int r) {
      return j0 + r < N ? k + ((j0 + r) * H_kv + g) * D : (const uint16_t*)nullptr;
    });
    load_rows(kIb + buf * (L::KI / 2), kWKeys, DI, k, [&](int r) {
      return j0 + r < N ? k_idx + (j0 + r) * DI : (const uint16_t*)nullptr;
    });
  };
  load_kt(0, 0);
  cp_async_commit();
  float lse_r[2], lseI_p[2];
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    const int64_t t = t0 + 2 * warp + ri;
    lse_r[ri] = (t < N && gq < gs) ? lse[(int64_t)(g * gs + gq) * N + t] : 0.f;
    lseI_p[ri] = t < N ? lseI[(int64_t)g * N + t] : 0.f;
  }
  float kl_acc[2] = {0.f, 0.f};
  float dq[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  const float sI = rsqrtf((float)DI);
  const uint32_t qs_a = smem_u32(Qs), qis_a = smem_u32(qIs), dz_a = smem_u32(dz_s);
  for (int kt = 0; kt < n_kt; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < n_kt) {
      load_kt(kt + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint32_t ks_a = smem_u32(Kb + buf * (L::K / 2)), kis_a = smem_u32(kIb + buf * (L::KI / 2));
    dz_tile<D, DI, true>(qs_a, qis_a, ks_a, kis_a, zI_s, dz_s, t0, (int64_t)kt * kWKeys, N, scale, sI, w_kl,
                         lse_r, lseI_p, gs, kl_acc);
    // dq^I (16 positions x columns 16w..16w+15) += dz (16 x 64) K^I (64 x d_I)
    if (16 * warp < DI) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t a[4], b[4];
        lds_a(a, dz_a, 0, 16 * kk, kWKeys);
        lds_b_kn(b, kis_a, 16 * kk, 16 * warp, DI);
        mma2(dq[0], dq[1], a, b);
      }
    }
    __syncthreads();
  }
  // KL of positions 2w, 2w+1 (terms spread over all lanes of the warp)
#pragma unroll
  for (int ri = 0; ri < 2; ++ri) {
    float x = kl_acc[ri];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    const int64_t t = t0 + 2 * warp + ri;
    if (lane == 0 && t < N) kl[(int64_t)g * N + t] = x;
  }
  if (16 * warp < DI) {
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
      for (int ri = 0; ri < 2; ++ri) {
        const int64_t t = t0 + gq + 8 * ri;
        if (t < N) {
          float* dst = dq_idx + (t * G + g) * DI + 16 * warp + 8 * n + 2 * tq;
          *reinterpret_cast<float2*>(dst) = make_float2(dq[n][2 * ri] * sI, dq[n][2 * ri + 1] * sI);
        }
      }
  }
}

// ------------------------------------------------------------------ dk
template <int D, int DI>
__global__ void __launch_bounds__(kWThreads, 1)
    warmup_dk_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                     const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ k_idx,
                     const float* __restrict__ lse, const float* __restrict__ lseI, int64_t N, int H_q, int H_kv,
                     float scale, float w_kl, float* __restrict__ dk_idx) {
  using L = WarmSmem<D, DI>;
  extern __shared__ __align__(128) uint8_t wsm[];
  uint16_t* Qb = reinterpret_cast<uint16_t*>(wsm);                               // [2][Q]
  uint16_t* qIb = reinterpret_cast<uint16_t*>(wsm + 2 * L::Q);                   // [2][QI]
  uint16_t* Ks = reinterpret_cast<uint16_t*>(wsm + 2 * L::Q + 2 * L::QI);
  uint16_t* kIs = reinterpret_cast<uint16_t*>(wsm + 2 * L::Q + 2 * L::QI + L::K);
  float* zI_s = reinterpret_cast<float*>(wsm + 2 * L::Q + 2 * L::QI + L::K + L::KI);
  uint16_t* dz_s = reinterpret_cast<uint16_t*>(wsm + 2 * L::Q + 2 * L::QI + L::K + L::KI + L::ZI);
  __shared__ float lse_s[2][kWRows], lseI_s[2][kWPos];
  const int G = H_kv, gs = H_q / H_kv;
  const int64_t n_kt = (N + kWKeys - 1) / kWKeys;
  const int64_t kt = (int64_t)blockIdx.x;  // key tiles in order: the first have the most query tiles
  const int g = blockIdx.y;
  const int64_t j0 = kt * kWKeys;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gq = lane >> 2, tq = lane & 3;
  const int64_t qt_first = j0 / kWPos, n_qt = (N + kWPos - 1) / kWPos;
  load_rows(Ks, kWKeys, D, k, [&](int r) {
    return j0 + r < N ? k + ((j0 + r) * H_kv + g) * D : (const uint16_t*)nullptr;
  });
  load_rows(kIs, kWKeys, DI, k, [&](int r) {
    return j0 + r < N ? k_idx + (j0 + r) * DI : (const uint16_t*)nullptr;
  });
  auto load_qt = [&](int64_t qt, int buf) {
    const int64_t t0 = qt * kWPos;
    load_rows(Qb + buf * (L::Q / 2), kWRows, D, q, [&](int r) { return q_row(q, t0, r, N, H_q, g, gs, D); });
    load_rows(qIb + buf * (L::QI / 2), kWPos, DI, q, [&](int r) {
      return t0 + r < N ? q_idx + ((t0 + r) * G + g) * DI : (const uint16_t*)nullptr;
    });
    for (int r = tid; r < kWRows; r += kWThreads) {
      const int64_t t = t0 + (r >> 3);
      const int hh = r & 7;
      lse_s[buf][r] = (t < N && hh < gs) ? lse[(int64_t)(g * gs + hh) * N + t] : 0.f;
    }
    for (int p = tid; p < kWPos; p += kWThreads) lseI_s[buf][p] = t0 + p < N ? lseI[(int64_t)g * N + t0 + p] : 0.f;
  };
  (void)n_kt;
  load_qt(qt_first, 0);
  cp_async_commit();
  // dk^I of keys 16 (w & 3).. x columns (w >> 2) * DI/2 ..: one k-step of 16 positions per query tile
  constexpr int NT = DI / 2 / 8;  // 8-column n-tiles per warp
  float dk[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) dk[n][0] = dk[n][1] = dk[n][2] = dk[n][3] = 0.f;
  const float sI = rsqrtf((float)DI);
  const uint32_t ks_a = smem_u32(Ks), kis_a = smem_u32(kIs), dz_a = smem_u32(dz_s);
  const int mt = warp & 3, ch = warp >> 2;
  for (int64_t qt = qt_first; qt < n_qt; ++qt) {
    const int buf = (int)((qt - qt_first) & 1);
    if (qt + 1 < n_qt) {
      __syncthreads();  // lse_s / lseI_s of buffer buf ^ 1 are no longer read
      load_qt(qt + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const int64_t t0 = qt * kWPos;
    const float lse_r[2] = {lse_s[buf][16 * warp + gq], lse_s[buf][16 * warp + gq + 8]};
    const float lseI_p[2] = {lseI_s[buf][2 * warp], lseI_s[buf][2 * warp + 1]};
    const uint32_t qs_a = smem_u32(Qb + buf * (L::Q / 2)), qis_a = smem_u32(qIb + buf * (L::QI / 2));
    float no_kl[2] = {0.f, 0.f};
    dz_tile<D, DI, false>(qs_a, qis_a, ks_a, kis_a, zI_s, dz_s, t0, j0, N, scale, sI, w_kl, lse_r, lseI_p, gs, no_kl);
    // dk^I (16 keys x DI/2 columns) += dz^T (keys x 16 positions) Q^I (16 positions x columns)
    uint32_t a[4];
    {
      // A = dz^T: 16 keys (rows) x 16 positions (k) from dz_s stored [position][key]
      const int mm = lane >> 3;
      ldsm_x4_t(a, tile_addr(dz_a, (lane & 7) + ((mm >> 1) << 3), 16 * mt + ((mm & 1) << 3), kWKeys));
    }
#pragma unroll
    for (int np = 0; np < NT / 2; ++np) {
      uint32_t b[4];
      lds_b_kn(b, qis_a, 0, ch * (DI / 2) + 16 * np, DI);
      mma2(dk[2 * np], dk[2 * np + 1], a, b);
    }
    __syncthreads();  // zI_s / dz_s are rewritten by the next tile
  }
  // fp32 reductions into dk_idx (the groups of a key tile add up there)
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      const int64_t j = j0 + 16 * mt + gq + 8 * ri;
      if (j < N) red_add2(dk_idx + j * DI + ch * (DI / 2) + 8 * n + 2 * tq, dk[n][2 * ri] * sI, dk[n][2 * ri + 1] * sI);
    }
}

template <int D, int DI>
cudaError_t launch_t(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx, int64_t N,
                     int H_q, int H_kv, float scale, float kl_weight, bool fwd, bool grad, void* out, float* lse,
                     float* lseI, float* dq_idx, float* dk_idx, float* kl, cudaStream_t s) {
  using L = WarmSmem<D, DI>;
  const int64_t n_qt = (N + kWPos - 1) / kWPos, n_kt = (N + kWKeys - 1) / kWKeys;
  const int fwd_smem = L::Q + L::QI + 4 * L::K + 2 * L::KI;
  const int dq_smem = L::Q + L::QI + 2 * L::K + 2 * L::KI + L::ZI + L::DZ;
  const int dk_smem = 2 * L::Q + 2 * L::QI + L::K + L::KI + L::ZI + L::DZ;
  cudaError_t e;
  if (fwd && warmup_tc_supported(D, DI, H_q, H_kv)) {  // dense attention and the index lse on the tensor cores
    if ((e = launch_warmup_fwd_tc(q, k, v, q_idx, k_idx, N, H_q, H_kv, scale, out, lse, lseI, nullptr, s)) !=
        cudaSuccess)
      return e;
  } else if (fwd) {
    if ((e = cudaFuncSetAttribute(warmup_fwd_kernel<D, DI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  fwd_smem)) != cudaSuccess)
      return e;
    warmup_fwd_kernel<D, DI><<<dim3((unsigned)n_qt, (unsigned)H_kv), kWThreads, fwd_smem, s>>>(
        (const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)v, (const uint16_t*)q_idx, (const uint16_t*)k_idx,
        N, H_q, H_kv, scale, (uint16_t*)out, lse, lseI);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (!grad) return cudaSuccess;
  if (warmup_tc_supported(D, DI, H_q, H_kv))  // one key-outer pass on the tensor cores
    return launch_warmup_grad_tc(q, k, q_idx, k_idx, N, H_q, H_kv, scale, kl_weight, lse, lseI, dq_idx, dk_idx, kl,
                                 nullptr, s);
  if ((e = cudaFuncSetAttribute(warmup_dq_kernel<D, DI>, cudaFuncAttributeMaxDynamicSharedMemorySize, dq_smem)) !=
      cudaSuccess)
    return e;
  warmup_dq_kernel<D, DI><<<dim3((unsigned)n_qt, (unsigned)H_kv), kWThreads, dq_smem, s>>>(
      (const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)q_idx, (const uint16_t*)k_idx, lse, lseI, N, H_q, H_kv,
      scale, kl_weight, dq_idx, kl);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dk_idx, 0, (size_t)N * DI * 4, s)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(warmup_dk_kernel<D, DI>, cudaFuncAttributeMaxDynamicSharedMemorySize, dk_smem)) !=
      cudaSuccess)
    return e;
  warmup_dk_kernel<D, DI><<<dim3((unsigned)n_kt, (unsigned)H_kv), kWThreads, dk_smem, s>>>(
      (const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)q_idx, (const uint16_t*)k_idx, lse, lseI, N, H_q, H_kv,
      scale, kl_weight, dk_idx);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_warmup(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx, int64_t N,
                          int H_q, int H_kv, int d, int d_I, float scale, float kl_weight, bool fwd, bool grad,
                          void* out, float* lse, float* lseI, float* dq_idx, float* dk_idx, float* kl, cudaStream_t s) {
  if (d == 64) {
    if (d_I == 32) return launch_t<64, 32>(q, k, v, q_idx, k_idx, N, H_q, H_kv, scale, kl_weight, fwd, grad, out, lse, lseI,
                                           dq_idx, dk_idx, kl, s);
    if (d_I == 64) return launch_t<64, 64>(q, k, v, q_idx, k_idx, N, H_q, H_kv, scale, kl_weight, fwd, grad, out, lse, lseI,
                                           dq_idx, dk_idx, kl, s);
    return launch_t<64, 128>(q, k, v, q_idx, k_idx, N, H_q, H_kv, scale, kl_weight, fwd, grad, out, lse, lseI, dq_idx, dk_idx,
                             kl, s);
  }
  if (d_I == 32) return launch_t<128, 32>(q, k, v, q_idx, k_idx, N, H_q, H_kv, scale, kl_weight, fwd, grad, out, lse, lseI,
                                          dq_idx, dk_idx, kl, s);
  if (d_I == 64) return launch_t<128, 64>(q, k, v, q_idx, k_idx, N, H_q, H_kv, scale, kl_weight, fwd, grad, out, lse, lseI,
                                          dq_idx, dk_idx, kl, s);
  return launch_t<128, 128>(q, k, v, q_idx, k_idx, N, H_q, H_kv, scale, kl_weight, fwd, grad, out, lse, lseI, dq_idx, dk_idx,
                            kl, s);
}

}  // namespace msa
