// msa_decode: one decode step for B sequences.
//
// velog llama.cpp analysis, section 2 (each step scans the whole 256 B/token
// index-key cache; the K/V read is fixed at the selected blocks) and section 4
// (block scores -> max-pooling -> forced local block + top-k -> attention over
// the selected blocks); "MSA" study note 2-3 for the equations.
//
// Two launches per step:
//   1. scan (+ merge): split-K over the cache, two 8-warp CTAs per SM.  Each
//      warp streams an equal share of 16-key chunks straight from HBM into
//      mma.sync A fragments (16-byte loads, one chunk (bf16) or three (E4M3)
//      in flight ahead of the one being scored; dims permuted consistently in the query fragments, so
//      no shared-memory staging is needed) and scores all groups at once
//      (16 keys x 8 groups x d_I per mma chain).  Block maxima meet in shared
//      memory (an atomic max on order-preserving integers joins the two parts
//      of a block split between warps); each CTA then writes its top-(k-1)
//      blocks per group as a list sorted best first (one warp-wide sort of
//      its blocks when it holds at most 128, else register lists popped in
//      k-1 rounds).
//   2. select + attend (+ combine): per (sequence, group, slot) one CTA merges
//      the group's lists up to its slot (every CTA of the group does the same
//      merge, from shared memory, so no single CTA holds the others up), reads
//      that block's K/V rows and produces each group head's partial (O, lse);
//      the last CTA of a (sequence, group) merges the k partials by their lse.
//      It is launched as a programmatic dependent of the scan, so its launch
//      overlaps the scan's tail.
#include <math.h>

#include <cudaTypedefs.h>
#include <mutex>

#include "msa_sm100.cuh"

namespace msa {

namespace {

constexpr int kScanThreads = 256;  // 8 warps, two CTAs per SM
constexpr int kScanWarps = kScanThreads / 32;
constexpr int kGroupsPerMma = 8;    // mma n = 8 groups
constexpr int kMergeListsPerLane = 8;  // list merge: splits <= 32 * 8
constexpr int kMaxCtaBlocks = 2048;     // block maxima kept in shared memory per scan CTA

// dims of fragment column kf (0..15) in k-step ks of the bf16 scan: see the load pattern below
__device__ __forceinline__ int frag_dim(int ks, int kf) {
  int p = ks >> 1, half = ks & 1;
  int c = (kf & 7) >> 1, e = kf & 1, hi = kf >> 3;
  return 32 * p + 8 * c + 4 * half + 2 * hi + e;
}
// the same for the E4M3 scan (m16n8k32: fragment column kf in 0..31, four codes per register)
__device__ __forceinline__ int frag_dim8(int ks, int kf) {
  int p = ks >> 1, half = ks & 1;
  int c = (kf & 15) >> 2, e = kf & 3, hi = kf >> 4;
  return 64 * p + 16 * c + 8 * half + 4 * hi + e;
}

// fp32 -> unsigned with the same order (-0 folded to +0); 0 is below every value
__device__ __forceinline__ uint32_t ordered_bits(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Completion ticket of the last-CTA pattern: __syncthreads gathers every
// thread's writes before thread 0 takes a ticket with acquire-release semantics
// at GPU scope (the release covers what the barrier ordered before it); the CTA
// that takes the last ticket reads the others' results after a __syncthreads
// (L2 loads only), which orders its reads after that acquire.
__device__ __forceinline__ unsigned int ticket_acq_rel(unsigned int* t) {
  unsigned int old;
  asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;\n" : "=r"(old) : "l"(t) : "memory");
  return old;
}

// The largest 64-bit key across the warp: two single-instruction reductions,
// the high words first, then the low words of the lanes that hold that high word.
__device__ __forceinline__ uint64_t warp_max_key(uint64_t x) {
  const uint32_t hi = (uint32_t)(x >> 32), lo = (uint32_t)x;
  const uint32_t mh = __reduce_max_sync(0xffffffffu, hi);
  const uint32_t ml = __reduce_max_sync(0xffffffffu, hi == mh ? lo : 0u);
  return ((uint64_t)mh << 32) | ml;
}

// Descending sort of the 32 R keys x[j] (element e = 32 j + lane) across a warp: a bitonic network whose
// partner at distance d is a shuffle for d < 32 and another register of the same lane for d >= 32.  In each
// compare-exchange the element with the lower index keeps the larger key exactly when its block of kk
// elements is to end up in descending order; the last merge (kk = 32 R) orders the whole warp.
template <int R>
__device__ __forceinline__ void warp_sort_desc(uint64_t (&x)[R], int lane) {
#pragma unroll
  for (int kk = 2; kk <= 32 * R; kk <<= 1) {
#pragma unroll
    for (int d = kk >> 1; d > 0; d >>= 1) {
      uint64_t y[R];
#pragma unroll
      for (int j = 0; j < R; ++j) {
        const int e = 32 * j + lane;
        uint64_t o;
        if (d >= 32) {
          o = x[j ^ (d >> 5)];
        } else {
          const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(x[j] >> 32), d);
          const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)x[j], d);
          o = ((uint64_t)hi << 32) | lo;
        }
        const bool keep_max = ((e & d) == 0) == ((e & kk) == 0);
        y[j] = keep_max == (x[j] > o) ? x[j] : o;
      }
#pragma unroll
      for (int j = 0; j < R; ++j) x[j] = y[j];
    }
  }
}

// 16-byte pieces 64q + 16c of key rows `row` and `row + 8` of a 16-key chunk (RB bytes per row)
template <int RB>
__device__ __forceinline__ void load_keys16(uint4 (&v)[RB / 64][2], const uint8_t* p) {
#pragma unroll
  for (int q = 0; q < RB / 64; ++q) {
    v[q][0] = ldg_stream_16(p + 64 * q);
    v[q][1] = ldg_stream_16(p + 8 * RB + 64 * q);
  }
}

// Scan CTA (split, seq): candidate blocks [b_lo, b_hi) of sequence seq, where
// the candidates are the blocks before the query's local block.  The CTA's
// 16-key chunks are divided evenly among its warps; a block whose chunks fall
// to two warps gets its maximum from both through the shared-memory atomic.
// F8: the index query and cache hold E4M3 codes; the same 16-byte pieces feed
// m16n8k32 E4M3 MMAs (32 dims per k-step instead of 16), so a key row is half
// the bytes and the scan reads half the cache traffic.
template <int DI, int BK, bool PAGED, bool F8, int CAP>
__global__ void __launch_bounds__(kScanThreads, 2) decode_scan_kernel(
    const uint8_t* __restrict__ q_idx_t, const uint8_t* __restrict__ k_idx_cache,
    const int32_t* __restrict__ ctx_len, int64_t ctx_max, CacheMap map, int G, int k, int splits,
    uint64_t* __restrict__ cand, DeviceStatus* st) {
  constexpr int RB = DI * (F8 ? 1 : 2);  // bytes per index row
  constexpr int NQ = RB / 64;            // 16-byte pieces per lane and row
  constexpr int KS = 2 * NQ;             // MMA k-steps per 16-key chunk
  static_assert(NQ >= 1, "index rows of at least 64 bytes");
  constexpr int CPB = BK / 16;  // chunks per block
  // [blocks of this CTA][8 groups], ordered_bits of the block maxima
  extern __shared__ __align__(16) uint32_t bmax_s[];
  griddep_launch_dependents();  // the attention grid may be scheduled once every scan CTA is resident
  const int seq = blockIdx.y, split = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = lane & 3, row = lane >> 2;
  const int km1 = k - 1;
  const int64_t len = ctx_len[seq];
  const bool ok = len >= 1 && len <= ctx_max;
  if (!ok && split == 0 && tid == 0) raise_error(st, kErrBadIndex, 2u);
  const int64_t t = ok ? len - 1 : 0;
  const int64_t local = t / BK;  // candidates: blocks [0, local)
  const int64_t b_lo = local * split / splits, b_hi = local * (split + 1) / splits;
  const int nblk = (int)(b_hi - b_lo);
  for (int i = tid; i < nblk * kGroupsPerMma; i += kScanThreads) bmax_s[i] = 0u;

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
          const uint8_t* qrow = q_idx_t + ((int64_t)seq * G + n) * RB;
          if (F8) {
#pragma unroll
            for (int e = 0; e < 4; ++e) w |= (uint32_t)qrow[frag_dim8(ks, 16 * r + 4 * c + e)] << (8 * e);
          } else {
            const uint16_t* qp = reinterpret_cast<const uint16_t*>(qrow);
            int d0 = frag_dim(ks, 2 * c + 8 * r), d1 = frag_dim(ks, 2 * c + 1 + 8 * r);
            w = (uint32_t)qp[d0] | ((uint32_t)qp[d1] << 16);
          }
        }
        qf[ks][r] = w;
      }
  }
  __syncthreads();

  // this warp's chunks [c0, c1) of the CTA's nblk * CPB.  Chunk indices and
  // offsets within the CTA's range are 32-bit (nblk <= kMaxCtaBlocks, so an
  // offset stays below 2^26 bytes): the per-chunk loop carries no 64-bit
  // integer arithmetic, which at E4M3's 2 KB chunks was most of its ALU work.
  constexpr int CPB_SHIFT = CPB == 8 ? 3 : CPB == 4 ? 2 : CPB == 2 ? 1 : 0;
  static_assert((1 << CPB_SHIFT) == CPB, "chunks per block is a power of two");
  const int nch = nblk * CPB;
  const int c0 = nch * warp / kScanWarps, c1 = nch * (warp + 1) / kScanWarps;
  const uint8_t* base = k_idx_cache + ((int64_t)seq * ctx_max + b_lo * BK + row) * RB + 16 * c;
  // first key row of chunk cc (+ row): contiguous, or through the page table (a page holds whole chunks)
  auto chunk_ptr = [&](int cc) -> const uint8_t* {
    if (!PAGED) return base + (uint32_t)cc * (uint32_t)(16 * RB);
    const int64_t key = b_lo * BK + (int64_t)cc * 16;
    const int64_t r = map.row(seq, key, st);
    return k_idx_cache + (r + row) * RB + 16 * c;
  };
  float bm0 = __int_as_float(0xff800000), bm1 = bm0;
  auto score = [&](const uint4 (&v)[NQ][2], int cc) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      // k-step 2q: bytes 0..7 of each lane's piece; k-step 2q+1: bytes 8..15
      const uint32_t a0[4] = {v[q][0].x, v[q][1].x, v[q][0].y, v[q][1].y};
      const uint32_t a1[4] = {v[q][0].z, v[q][1].z, v[q][0].w, v[q][1].w};
      if (F8) {
        mma_e4m3_16832(acc, a0, qf[2 * q]);
        mma_e4m3_16832(acc, a1, qf[2 * q + 1]);
      } else {
        mma_bf16_16816(acc, a0, qf[2 * q]);
        mma_bf16_16816(acc, a1, qf[2 * q + 1]);
      }
    }
    bm0 = fmaxf(bm0, fmaxf(acc[0], acc[2]));  // group 2c, keys row and row+8
    bm1 = fmaxf(bm1, fmaxf(acc[1], acc[3]));  // group 2c+1
    if ((cc & (CPB - 1)) == CPB - 1 || cc == c1 - 1) {  // end of this warp's part of a block
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, o));
        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, o));
      }
      // group g's maximum sits in lane g/2 (value g&1)
      const float x0 = __shfl_sync(0xffffffffu, bm0, (lane & 7) >> 1);
      const float x1 = __shfl_sync(0xffffffffu, bm1, (lane & 7) >> 1);
      if (lane < G) atomicMax(&bmax_s[(cc >> CPB_SHIFT) * kGroupsPerMma + lane], ordered_bits((lane & 1) ? x1 : x0));
      bm0 = bm1 = __int_as_float(0xff800000);
    }
  };
  // a ring of PD chunks: PD - 1 in flight ahead of the one being scored (about 4-6 KB per warp either way)
  constexpr int PD = F8 ? 4 : 2;
  uint4 vr[PD][NQ][2];
#pragma unroll
  for (int p = 0; p < PD - 1; ++p)
    if (c0 + p < c1) load_keys16<RB>(vr[p], chunk_ptr(c0 + p));
  for (int ci = c0; ci < c1; ci += PD) {
#pragma unroll
    for (int p = 0; p < PD; ++p) {
      const int cc = ci + p;
      if (cc < c1) {
        if (cc + PD - 1 < c1) load_keys16<RB>(vr[(p + PD - 1) % PD], chunk_ptr(cc + PD - 1));
        score(vr[p], cc);
      }
    }
  }
  __syncthreads();

  // this CTA's top-(k-1) blocks of group g (warp g), best first (0 where the CTA has fewer candidates).
  // Up to 128 blocks: one warp-wide sort of their (maximum, ~id) keys.  More: lane l ranks blocks l,
  // l + 32, ... into its register list of the best CAP (one insertion site in a rolled loop), then k-1
  // rounds of a warp-wide maximum over the lists' heads pop the CTA's list.
  const int kp = km1 + (km1 & 1);  // list stride: an even count of keys (16-byte rows)
  if (warp < G && nblk <= 128) {
    const int g = warp;
    uint64_t x[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int b = 32 * j + lane;
      const uint32_t o = b < nblk ? bmax_s[b * kGroupsPerMma + g] : 0u;
      x[j] = o ? ((uint64_t)o << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)(b_lo + b)) : 0ull;
    }
    warp_sort_desc<4>(x, lane);
    uint64_t* out = cand + (((int64_t)seq * G + g) * splits + split) * kp;
    if (lane < km1) out[lane] = x[0];  // k - 1 <= 32
  } else if (warp < G) {
    const int g = warp;
    TopK<CAP> top;
    top.init(CAP);
#pragma unroll 1
    for (int b = lane; b < nblk; b += 32) {
      const uint32_t o = bmax_s[b * kGroupsPerMma + g];
      if (o) top.insert_key(((uint64_t)o << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)(b_lo + b)));
    }
    uint64_t* out = cand + (((int64_t)seq * G + g) * splits + split) * kp;
    for (int r = 0; r < km1; ++r) {
      const uint64_t best = warp_max_key(top.key[CAP - 1]);
      const bool pop = best != 0ull && top.key[CAP - 1] == best;  // keys are unique: one lane pops
#pragma unroll
      for (int i = CAP - 1; i > 0; --i) top.key[i] = pop ? top.key[i - 1] : top.key[i];
      top.key[0] = pop ? 0ull : top.key[0];
      if (lane == 0) out[r] = best;  // 0 = no candidate
    }
  }
}

// The r-th best key (r >= 1) over `splits` lists of km1 keys (stride kp),
// each sorted best first, staged in shared memory; one warp, lane l holding
// lists l, l + 32, ... (LPL of them).  Each round takes the warp's best head
// and advances that list.  The list's next key sits in a register, loaded one
// round ahead, so a round waits on no shared-memory load; the advance is
// branch-free, so the warp never splits over the lane that owns the winner.
template <int LPL>
__device__ __forceinline__ uint64_t merged_key(const uint64_t* sl, int splits, int kp, int km1, int r, int lane) {
  uint64_t head[LPL], nxt[LPL];
  int pos[LPL];
#pragma unroll
  for (int i = 0; i < LPL; ++i) {
    const int sp = lane + 32 * i;
    const bool in = sp < splits;
    pos[i] = 0;
    head[i] = in && km1 > 0 ? sl[sp * kp] : 0ull;
    nxt[i] = in && km1 > 1 ? sl[sp * kp + 1] : 0ull;
  }
  uint64_t best = 0ull;
  for (int j = 0; j < r; ++j) {
    uint64_t m[LPL];  // the lane's best head, as a tree
#pragma unroll
    for (int i = 0; i < LPL; ++i) m[i] = head[i];
#pragma unroll
    for (int w = LPL / 2; w >= 1; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) m[i] = m[i] > m[i + w] ? m[i] : m[i + w];
    best = warp_max_key(m[0]);
    if (best == 0ull) break;  // fewer candidates than r (uniform: the reduction's result)
#pragma unroll
    for (int i = 0; i < LPL; ++i) {
      const bool hit = head[i] == best;  // keys are unique: block ids differ across lists
      pos[i] += hit ? 1 : 0;
      const uint64_t nn = hit && pos[i] + 1 < km1 ? sl[(lane + 32 * i) * kp + pos[i] + 1] : 0ull;
      head[i] = hit ? nxt[i] : head[i];
      nxt[i] = hit ? nn : nxt[i];
    }
  }
  return best;
}

// One CTA (4 warps) per (slot, group, sequence).  Its block: slot 0 is the
// local block; slot r + 1 is the r-th best candidate over the scan CTAs'
// lists of the group (merged_key over the lists staged in shared memory).  The
// CTA writes its slot of block_idx.  The group's heads are the rows of m16n8k16 tensor-core tiles
// (rows >= gs are zero) and warp w takes keys [w BK/4, (w+1) BK/4):
//   - K rows go straight from HBM into B fragments (16-byte loads; the head
//     dims are permuted the same way in the query's A fragments, as in the
//     scan), so only V is staged in shared memory (16-byte chunk c of row j
//     stored at chunk c ^ (j mod d/8), so ldmatrix rows fall in distinct
//     banks), which keeps every CTA of the grid resident at once;
//   - the softmax statistics are merged across warps in shared memory, P stays
//     in registers as the A operand of P V (V read transposed by ldmatrix),
//     and the warps' partial O are summed in shared memory before the head's
//     partial (O, lse) is written.
// The last CTA of a (sequence, group) to finish merges the group's k partials
// per head: M = max lse_s, w_s = e^(lse_s - M) / sum e^(lse_s - M),
// out = sum w_s O_s, lse = M + ln sum e^(lse_s - M).
template <int D, int BK, bool PAGED, int LPL>
__global__ void __launch_bounds__(128) decode_attn_kernel(const uint16_t* __restrict__ q_t,
                                                          const uint16_t* __restrict__ k_cache,
                                                          const uint16_t* __restrict__ v_cache,
                                                          const int32_t* __restrict__ ctx_len,
                                                          const uint64_t* __restrict__ cand, int splits,
                                                          int32_t* __restrict__ block_idx, int64_t ctx_max,
                                                          CacheMap map, int H_q, int G, int k, float scale,
                                                          float* __restrict__ part_o, float* __restrict__ part_lse,
                                                          unsigned int* __restrict__ tickets,
                                                          uint16_t* __restrict__ out, float* __restrict__ lse,
                                                          DeviceStatus* st) {
  // the group's candidate lists first; then V rows [BK][D]; later the warps' partial O
  extern __shared__ __align__(16) uint16_t v_s[];
  __shared__ float red_m[4][8], red_l[4][8];
  __shared__ float w_s[8][32];  // combine weights [head][slot]
  __shared__ int s_last;
  __shared__ int32_t s_blk;
  __shared__ int64_t krow_s[PAGED ? BK : 1];  // cache row of each key of the block (paged caches)
  constexpr int C8 = D / 8;     // 16-byte chunks per row
  constexpr int KPW = BK / 4;   // keys per warp
  constexpr int NT = KPW / 8;   // 8-key n-tiles per warp
  constexpr int NP = D / 32;    // 16-byte pieces of a row per lane (two k-steps over d each)
  static_assert(NT % 2 == 0, "P V k-steps take two n-tiles");
  static_assert(4 * 8 * D * 4 <= BK * D * 2, "partial O sums fit over V");
  const int slot = blockIdx.x, g = blockIdx.y, seq = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = lane >> 2, tq = lane & 3;  // fragment row (head; key of a B column) and column pair
  const int gs = H_q / G;
  const int64_t len = ctx_len[seq];
  // q as A fragments: row gq = head gq of the group (zero past gs), rows 8..15 zero; piece p holds dims
  // 32p + 8tq .. +7: words x, y feed k-step 2p and z, w k-step 2p+1 (the order of the K fragments below)
  uint4 qv[NP];
  {
    const uint16_t* qrow = q_t + ((int64_t)seq * H_q + g * gs + gq) * D + 8 * tq;
#pragma unroll
    for (int p = 0; p < NP; ++p) qv[p] = gq < gs ? ldg_stream_16(qrow + 32 * p) : make_uint4(0u, 0u, 0u, 0u);
  }
  const bool ok = len >= 1 && len <= ctx_max;
  griddep_wait();  // the candidate lists come from the scan grid
  if (slot == 0) {
    if (tid == 0) s_blk = ok ? (int32_t)((len - 1) / BK) : -1;
  } else {
    const int kp = (k - 1) + ((k - 1) & 1);  // list stride (an even count of keys)
    const uint64_t* gl = cand + (((int64_t)seq * G + g) * splits) * kp;
    uint64_t* sl = reinterpret_cast<uint64_t*>(v_s);
    const int n16 = splits * kp / 2;  // 16-byte pieces
    for (int i = tid; i < n16; i += blockDim.x) cp_async_16(sl + 2 * i, gl + 2 * i, 16);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    if (warp == 0) {
      const uint64_t best = merged_key<LPL>(sl, splits, kp, k - 1, slot, lane);
      if (lane == 0) s_blk = best ? (int32_t)(0xFFFFFFFFu - (uint32_t)best) : -1;
    }
  }
  __syncthreads();  // s_blk, and the lists are no longer read: v_s takes the V rows
  const int32_t b = s_blk;
  if (tid == 0) block_idx[((int64_t)seq * G + g) * k + slot] = b;
  const int64_t nb = (ctx_max + BK - 1) / BK;
  const bool valid = ok && b >= 0 && (int64_t)b < nb;
  const int64_t t = len - 1;
  const int64_t key0 = (int64_t)b * BK;
  const int nvis = valid ? (int)max((int64_t)0, min((int64_t)BK, t - key0 + 1)) : 0;
  float* po = part_o + (((int64_t)seq * H_q + g * gs) * k + slot) * D;
  float* pl = part_lse + ((int64_t)seq * H_q + g * gs) * k + slot;
  if (nvis == 0) {
    for (int hh = tid; hh < gs; hh += blockDim.x) pl[(int64_t)hh * k] = __int_as_float(0xff800000);
  } else {
    const int64_t kv_row = (int64_t)G * D;
    // key j of the block: row key0 + j of this sequence's cache, or row krow_s[j] of the page pool
    const int64_t first = PAGED ? 0 : (int64_t)seq * ctx_max + key0;
    const uint16_t* Kb = k_cache + first * kv_row + (int64_t)g * D;
    const uint16_t* Vb = v_cache + first * kv_row + (int64_t)g * D;
    if (PAGED) {
      for (int j = tid; j < BK; j += blockDim.x) krow_s[j] = j < nvis ? map.row(seq, key0 + j, st) : 0;
      __syncthreads();
    }
    auto row_off = [&](int j) -> int64_t { return (PAGED ? krow_s[PAGED ? j : 0] : (int64_t)j) * kv_row; };
    // V rows into shared memory (rows past nvis read as zero), every copy in flight at once
    for (int i = tid; i < BK * C8; i += blockDim.x) {
      const int j = i / C8, c8 = i % C8;
      const bool in = j < nvis;
      cp_async_16(v_s + j * D + (c8 ^ (j & (C8 - 1))) * 8, Vb + row_off(in ? j : 0) + c8 * 8, in ? 16 : 0);
    }
    cp_async_commit();
    // K rows of this warp's keys as B fragments (key = column gq of n-tile nt); rows past nvis repeat a
    // visible row and are masked below
    uint4 kf[NT][NP];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int j = min(warp * KPW + nt * 8 + gq, nvis - 1);
      const uint16_t* kr = Kb + row_off(j) + 8 * tq;
#pragma unroll
      for (int p = 0; p < NP; ++p) kf[nt][p] = ldg_stream_16(kr + 32 * p);
    }
    // S = q K^T for this warp's keys
    float sacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const uint32_t a0[4] = {qv[p].x, 0u, qv[p].y, 0u};
      const uint32_t a1[4] = {qv[p].z, 0u, qv[p].w, 0u};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint32_t b0[2] = {kf[nt][p].x, kf[nt][p].y}, b1[2] = {kf[nt][p].z, kf[nt][p].w};
        mma_bf16_16816(sacc[nt], a0, b0);
        mma_bf16_16816(sacc[nt], a1, b1);
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
    cp_async_wait<0>();
    __syncthreads();
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
        ldmatrix_x4_trans(r0, r1, r2, r3, v_s + key * D + ((chunk ^ (key & (C8 - 1))) * 8));
        const uint32_t b0[2] = {r0, r1}, b1[2] = {r2, r3};
        mma_bf16_16816(oacc[nd], a, b0);
        mma_bf16_16816(oacc[nd + 1], a, b1);
      }
    }
    // sum the warps' partial O in shared memory (over the V rows, which are no longer read)
    __syncthreads();
    float* red_o = reinterpret_cast<float*>(v_s);  // [4 warps][8 rows][D]
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
  }  // nvis > 0

  // the last of the group's k CTAs merges the partials
  __syncthreads();
  if (tid == 0) s_last = ticket_acq_rel(&tickets[(int64_t)seq * G + g]) == (unsigned)(k - 1);
  __syncthreads();
  if (!s_last) return;
  const float* gl = part_lse + ((int64_t)seq * H_q + g * gs) * k;  // [gs][k]
  // one warp per head, lane = slot (k <= 32): M, the weights and L by warp reductions
  for (int hh = warp; hh < gs; hh += blockDim.x / 32) {
    const float v = lane < k ? __ldcg(gl + hh * k + lane) : __int_as_float(0xff800000);
    float M = v;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w = M == __int_as_float(0xff800000) || v == __int_as_float(0xff800000) ? 0.f : __expf(v - M);
    float L = w;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    w_s[hh][lane] = w * inv;
    if (lane == 0 && lse)
      lse[(int64_t)seq * H_q + g * gs + hh] = L > 0.f ? M + logf(L) : __int_as_float(0xff800000);
  }
  __syncthreads();
  // thread -> (head, 4 columns); the partial loads of 16 slots are all in flight before the sums
  const float* go = part_o + ((int64_t)seq * H_q + g * gs) * k * D;  // [gs][k][D]
  for (int i = tid; i < gs * (D / 4); i += blockDim.x) {
    const int hh = i / (D / 4), dc = 4 * (i % (D / 4));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < k; s0 += 16) {
      float4 o[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int s = s0 + j;
        const bool use = s < k && w_s[hh][s < k ? s : 0] != 0.f;
        o[j] = use ? __ldcg(reinterpret_cast<const float4*>(go + ((int64_t)hh * k + s) * D + dc))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int s = s0 + j;
        const float w = s < k ? w_s[hh][s] : 0.f;
        acc.x += w * o[j].x;
        acc.y += w * o[j].y;
        acc.z += w * o[j].z;
        acc.w += w * o[j].w;
      }
    }
    const uint32_t lo = pack_bf16x2(acc.x, acc.y), hi = pack_bf16x2(acc.z, acc.w);
    uint16_t* o = out + ((int64_t)seq * H_q + g * gs + hh) * D + dc;  // out needs only 2-byte alignment
    o[0] = (uint16_t)(lo & 0xFFFFu);
    o[1] = (uint16_t)(lo >> 16);
    o[2] = (uint16_t)(hi & 0xFFFFu);
    o[3] = (uint16_t)(hi >> 16);
  }
  if (tid == 0) tickets[(int64_t)seq * G + g] = 0u;  // ready for the next call
}


struct DecodeScratch {
  unsigned int* tickets;  // [B * G] attention; cleared before every call
  uint64_t* cand;         // [B, G, splits, kp] per-CTA candidate keys (kp = k-1 rounded up to even)
  int32_t* blk;
  float* part_o;
  float* part_lse;
};

static size_t ticket_bytes(const DecodePlan& p) { return align_up((size_t)p.B * p.H_kv * 4, 256); }
static int list_stride(const DecodePlan& p) { return p.k > 1 ? (p.k - 1) + ((p.k - 1) & 1) : 2; }
// one group's lists, staged in shared memory by each attention CTA (at most 256 splits x 32 keys = 64 KB)
static size_t group_lists_bytes(const DecodePlan& p) { return (size_t)p.splits * list_stride(p) * 8; }

static size_t carve(const DecodePlan& p, void* base, DecodeScratch* out) {
  char* c = (char*)base;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* r = c ? c + off : nullptr;
    off += align_up(bytes, 256);
    return r;
  };
  DecodeScratch s;
  s.tickets = (unsigned int*)take(ticket_bytes(p));
  s.cand = (uint64_t*)take((size_t)p.B * p.splits * p.H_kv * list_stride(p) * 8);
  s.blk = (int32_t*)take((size_t)p.B * p.H_kv * p.k * 4);
  s.part_o = (float*)take((size_t)p.B * p.H_q * p.k * p.d * 4);
  s.part_lse = (float*)take((size_t)p.B * p.H_q * p.k * 4);
  if (out) *out = s;
  return off;
}

template <int DI, int BK, bool PAGED, bool F8, int CAP>
cudaError_t launch_scan_c(const void* q_idx_t, const void* k_idx_cache, const int32_t* ctx_len, const CacheMap& map,
                          const DecodePlan& p, const DecodeScratch& sc, DeviceStatus* st,
                          cudaStream_t s) {
  const size_t smem = (size_t)p.max_cta_blocks * kGroupsPerMma * 4;
  auto kern = decode_scan_kernel<DI, BK, PAGED, F8, CAP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3((unsigned)p.splits, (unsigned)p.B), kScanThreads, smem, s>>>(
      (const uint8_t*)q_idx_t, (const uint8_t*)k_idx_cache, ctx_len, p.ctx_max, map, p.H_kv, p.k, p.splits, sc.cand,
      st);
  return cudaGetLastError();
}

template <int DI, int BK, bool PAGED, bool F8>
cudaError_t launch_scan_t(const void* q_idx_t, const void* k_idx_cache, const int32_t* ctx_len, const CacheMap& map,
                          const DecodePlan& p, const DecodeScratch& sc, DeviceStatus* st,
                          cudaStream_t s) {
  return p.k - 1 <= 16 ? launch_scan_c<DI, BK, PAGED, F8, 16>(q_idx_t, k_idx_cache, ctx_len, map, p, sc, st, s)
                       : launch_scan_c<DI, BK, PAGED, F8, 32>(q_idx_t, k_idx_cache, ctx_len, map, p, sc, st, s);
}

template <int DI, int BK>
cudaError_t launch_scan(const void* q_idx_t, const void* k_idx_cache, const int32_t* ctx_len, const CacheMap& map,
                        const DecodePlan& p, const DecodeScratch& sc, DeviceStatus* st, cudaStream_t s) {
  if constexpr (DI >= 64) {  // E4M3 rows of 64 or 128 bytes
    if (p.f8)
      return map.table ? launch_scan_t<DI, BK, true, true>(q_idx_t, k_idx_cache, ctx_len, map, p, sc, st, s)
                       : launch_scan_t<DI, BK, false, true>(q_idx_t, k_idx_cache, ctx_len, map, p, sc, st, s);
  } else {
    if (p.f8) return cudaErrorInvalidValue;
  }
  return map.table ? launch_scan_t<DI, BK, true, false>(q_idx_t, k_idx_cache, ctx_len, map, p, sc, st, s)
                   : launch_scan_t<DI, BK, false, false>(q_idx_t, k_idx_cache, ctx_len, map, p, sc, st, s);
}

// The attention grid as a programmatic dependent of the scan: its CTAs may be
// scheduled while the scan drains and wait (griddepcontrol.wait) for its results.
template <int D, int BK, bool PAGED, int LPL>
cudaError_t launch_attn_dep_t(const void* q_t, const void* k_cache, const void* v_cache, const int32_t* ctx_len,
                              int32_t* blk, const CacheMap& map, const DecodePlan& p, float scale,
                              const DecodeScratch& sc, void* out, float* lse, DeviceStatus* st, cudaStream_t s) {
  const size_t vb = (size_t)BK * D * 2, lb = group_lists_bytes(p);
  const int smem = (int)(vb > lb ? vb : lb);  // V rows of one block, or first the group's candidate lists
  auto kern = decode_attn_kernel<D, BK, PAGED, LPL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.k, (unsigned)p.H_kv, (unsigned)p.B);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, (const uint16_t*)q_t, (const uint16_t*)k_cache, (const uint16_t*)v_cache,
                            ctx_len, (const uint64_t*)sc.cand, p.splits, blk, p.ctx_max, map, p.H_q, p.H_kv, p.k,
                            scale, sc.part_o, sc.part_lse, sc.tickets, (uint16_t*)out, lse, st);
}

template <int D, int BK, bool PAGED>
cudaError_t launch_attn_dep_p(const void* q_t, const void* k_cache, const void* v_cache, const int32_t* ctx_len,
                              int32_t* blk, const CacheMap& map, const DecodePlan& p, float scale,
                              const DecodeScratch& sc, void* out, float* lse, DeviceStatus* st, cudaStream_t s) {
  // lists per lane of the merge: splits <= 64, 128, 256
  if (p.splits <= 64)
    return launch_attn_dep_t<D, BK, PAGED, 2>(q_t, k_cache, v_cache, ctx_len, blk, map, p, scale, sc, out, lse, st, s);
  if (p.splits <= 128)
    return launch_attn_dep_t<D, BK, PAGED, 4>(q_t, k_cache, v_cache, ctx_len, blk, map, p, scale, sc, out, lse, st, s);
  return launch_attn_dep_t<D, BK, PAGED, 8>(q_t, k_cache, v_cache, ctx_len, blk, map, p, scale, sc, out, lse, st, s);
}

template <int D, int BK>
cudaError_t launch_attn_dep(const void* q_t, const void* k_cache, const void* v_cache, const int32_t* ctx_len,
                            int32_t* blk, const CacheMap& map, const DecodePlan& p, float scale,
                            const DecodeScratch& sc, void* out, float* lse, DeviceStatus* st, cudaStream_t s) {
  return map.table ? launch_attn_dep_p<D, BK, true>(q_t, k_cache, v_cache, ctx_len, blk, map, p, scale, sc, out, lse,
                                                     st, s)
                   : launch_attn_dep_p<D, BK, false>(q_t, k_cache, v_cache, ctx_len, blk, map, p, scale, sc, out,
                                                      lse, st, s);
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
  const int64_t cand_max = ctx_max >= 1 ? (ctx_max - 1) / Bk : 0;  // candidate blocks of the longest sequence
  int64_t splits = ((int64_t)num_sms() * 2 + B - 1) / B;           // two scan CTAs per SM
  const int64_t few = cand_max / 8 > 1 ? cand_max / 8 : 1;          // at least ~8 blocks per CTA
  if (splits > few) splits = few;
  const int64_t need = (cand_max + kMaxCtaBlocks - 1) / kMaxCtaBlocks;  // shared-memory bound per CTA
  if (splits < need) splits = need;
  if (splits > 32 * kMergeListsPerLane) splits = 32 * kMergeListsPerLane;
  if (splits < 1) splits = 1;
  p.splits = (int)splits;
  p.max_cta_blocks = (int)((cand_max + splits - 1) / splits);
  if (p.max_cta_blocks < 1) p.max_cta_blocks = 1;
  return p;
}

size_t decode_scratch_bytes(const DecodePlan& p) { return carve(p, nullptr, nullptr); }

size_t decode_clear_bytes(const DecodePlan& p) { return ticket_bytes(p); }

cudaError_t launch_decode(const void* q_t, const void* q_idx_t, const void* k_idx_cache, const void* k_cache,
                          const void* v_cache, const int32_t* ctx_len, const DecodePlan& p, float scale, void* out,
                          float* lse, int32_t* block_idx, void* scratch, DeviceStatus* st, cudaStream_t s,
                          const CacheMap* paged) {
  const CacheMap map = paged ? *paged : CacheMap{};
  DecodeScratch sc;
  carve(p, scratch, &sc);
  int32_t* blk = block_idx ? block_idx : sc.blk;
  cudaError_t e;
  if (p.d_I == 32) {
    e = p.Bk == 64 ? launch_scan<32, 64>(q_idx_t, k_idx_cache, ctx_len, map, p, sc, st, s)
                   : launch_scan<32, 128>(q_idx_t, k_idx_cache, ctx_len, map, p, sc, st, s);
  } else if (p.d_I == 64) {
    e = p.Bk == 64 ? launch_scan<64, 64>(q_idx_t, k_idx_cache, ctx_len, map, p, sc, st, s)
                   : launch_scan<64, 128>(q_idx_t, k_idx_cache, ctx_len, map, p, sc, st, s);
  } else {
    e = p.Bk == 64 ? launch_scan<128, 64>(q_idx_t, k_idx_cache, ctx_len, map, p, sc, st, s)
                   : launch_scan<128, 128>(q_idx_t, k_idx_cache, ctx_len, map, p, sc, st, s);
  }
  if (e != cudaSuccess) return e;
  if (p.d == 64)
    return p.Bk == 64 ? launch_attn_dep<64, 64>(q_t, k_cache, v_cache, ctx_len, blk, map, p, scale, sc, out, lse, st, s)
                      : launch_attn_dep<64, 128>(q_t, k_cache, v_cache, ctx_len, blk, map, p, scale, sc, out, lse, st, s);
  return p.Bk == 64 ? launch_attn_dep<128, 64>(q_t, k_cache, v_cache, ctx_len, blk, map, p, scale, sc, out, lse, st, s)
                    : launch_attn_dep<128, 128>(q_t, k_cache, v_cache, ctx_len, blk, map, p, scale, sc, out, lse, st, s);
}

// ---------------------------------------------------------------- fixed scratch for msa_decode_noalloc
// Scratch of the decode step for callers that cannot allocate device memory:
// a file-scope device array, resident on every GPU that loads the library
// until the process exits.  In host code `g_noalloc_scratch` names a host-side
// shadow, not device memory, so kernels only ever receive the address looked
// up below with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Unique id of the calling thread's current context (cuCtxGetId), 0 when none is
// current.  The driver calls come through the runtime's entry-point table, so
// the library links no libcuda.
static cudaError_t current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  *id = 0;
  if (!get_current || !get_id) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 4000, cudaEnableDefault, &q1) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || !f1)
      return cudaErrorNotSupported;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess || !f2)
      return cudaErrorNotSupported;
    get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f1);
    get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f2);
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
  if (!ctx) return cudaSuccess;
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

// The array's device address is looked up once per device and context, with
// that device current: after cudaDeviceReset, or with another context made
// current, the module is loaded again and the address is looked up again
// (context ids are never reused within a process).
cudaError_t noalloc_scratch(size_t need, void** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  static unsigned long long ctx_of[kMaxDevices] = {};
  *out = nullptr;
  if (need > kNoAllocScratchBytes) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long id = 0;
  e = current_context_id(&id);
  if (e != cudaSuccess) return e;
  if (!addr[dev] || id == 0 || ctx_of[dev] != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // makes the device's context current if none was
    if (e != cudaSuccess) return e;
    e = current_context_id(&id);
    if (e != cudaSuccess) return e;
    if (id == 0) return cudaErrorInvalidResourceHandle;
    addr[dev] = p;
    ctx_of[dev] = id;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace msa
