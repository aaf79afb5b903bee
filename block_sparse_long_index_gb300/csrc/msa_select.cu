// msa_select_blocks: index scoring + block max-pooling + local-pinned top-k.
//
// "MSA" study note 2-3 (s = q^I.k^I / sqrt(d_I); S = max over the block's
// tokens j <= t; set = local block + top-k), 3-2 (max-pooling), 3-5
// (exp-free top-k on raw scores) and Flash-MSA "プロキシアテンション"
// (per-tile maxima inserted into a register top-k while sweeping keys; local
// block pinned).
//
// One CTA owns 128 consecutive query rows of one group.  Their index queries
// stay in registers as MMA fragments; index-key tiles of 64 keys stream
// through a double-buffered shared-memory ring.  A tile's 128x64 raw scores
// live only in accumulator registers: each row takes its maximum over the
// tile, folds it into the running block maximum and, at the end of a block,
// offers (max, block) to a per-row top-(k-1) list held in registers.  No score
// is ever written to memory.  Only blocks b < local(t) are candidates: for
// every such block all its tokens satisfy j <= t, so no causal mask is
// needed, and the local block is emitted directly as slot 0.
#include "msa_common.cuh"

namespace msa {

namespace {

constexpr int kRows = 128;   // query rows per CTA
constexpr int kKeys = 64;    // keys per streamed tile
constexpr int kThreads = 128;

template <int DI, int BK, int CAP>
__global__ void __launch_bounds__(kThreads) select_kernel(const uint16_t* __restrict__ q_idx,
                                                          const uint16_t* __restrict__ k_idx, int64_t N, int G,
                                                          int k, int32_t* __restrict__ block_idx) {
  constexpr int LDS = DI + 8;  // padded row (elements): ldmatrix rows hit distinct banks
  constexpr int KS = DI / 16;  // MMA k-steps
  extern __shared__ __align__(16) uint16_t smem[];
  uint16_t* Qs = smem;                  // [kRows][LDS]
  uint16_t* Ks = smem + kRows * LDS;    // [2][kKeys][LDS]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.y;
  const int64_t n_tiles = (N + kRows - 1) / kRows;
  const int64_t r0 = (n_tiles - 1 - (int64_t)blockIdx.x) * kRows;  // longest rows first
  const int64_t t_last = min(r0 + kRows - 1, N - 1);
  const int64_t n_kt = (t_last / BK) * BK / kKeys;  // key tiles before the last row's block

  // ---- index queries of the CTA's rows (zero rows past N)
  for (int i = tid; i < kRows * (DI / 8); i += kThreads) {
    int r = i / (DI / 8), c8 = i % (DI / 8);
    int64_t t = r0 + r;
    int64_t tc = t < N ? t : N - 1;
    cp_async_16(Qs + r * LDS + c8 * 8, q_idx + (tc * G + g) * DI + c8 * 8, t < N ? 16 : 0);
  }
  cp_async_commit();

  auto load_keys = [&](int64_t kt, int buf) {
    uint16_t* dst = Ks + buf * kKeys * LDS;
    for (int i = tid; i < kKeys * (DI / 8); i += kThreads) {
      int r = i / (DI / 8), c8 = i % (DI / 8);
      cp_async_16(dst + r * LDS + c8 * 8, k_idx + (kt * kKeys + r) * DI + c8 * 8, 16);
    }
    cp_async_commit();
  };
  if (n_kt > 0) load_keys(0, 0);

  // owner row of this thread: quad lane c owns (m-tile c>>1, half c&1)
  const int c = lane & 3;
  const int64_t t_own = r0 + warp * 32 + 16 * (c >> 1) + 8 * (c & 1) + (lane >> 2);
  const int64_t local_own = t_own / BK;

  TopK<CAP> top;
  top.init(k - 1);
  float run = __int_as_float(0xff800000);

  if (n_kt > 0) {
    cp_async_wait<1>();
    __syncthreads();
  } else {
    cp_async_wait<0>();
    __syncthreads();
  }
  uint32_t qf[2][KS][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const uint16_t* p = Qs + (warp * 32 + mt * 16 + (lane & 15)) * LDS + ks * 16 + 8 * (lane >> 4);
      ldmatrix_x4(qf[mt][ks][0], qf[mt][ks][1], qf[mt][ks][2], qf[mt][ks][3], p);
    }

  for (int64_t kt = 0; kt < n_kt; ++kt) {
    if (kt + 1 < n_kt) {
      load_keys(kt + 1, (int)((kt + 1) & 1));
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint16_t* Kb = Ks + (int)(kt & 1) * kKeys * LDS;

    float acc[2][kKeys / 8][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < kKeys / 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;

#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int np = 0; np < kKeys / 16; ++np) {
        uint32_t b0[2], b1[2];
        const uint16_t* p = Kb + (np * 16 + (lane & 7) + 8 * (lane >> 4)) * LDS + ks * 16 + 8 * ((lane >> 3) & 1);
        ldmatrix_x4(b0[0], b0[1], b1[0], b1[1], p);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          mma_bf16_16816(acc[mt][2 * np], qf[mt][ks], b0);
          mma_bf16_16816(acc[mt][2 * np + 1], qf[mt][ks], b1);
        }
      }
    }
    __syncthreads();  // the buffer just read is refilled by the next prefetch

    // row maxima of the tile: quad-local max over the thread's columns, then across the quad
    float rm[2][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float m = fmaxf(acc[mt][0][2 * h], acc[mt][0][2 * h + 1]);
#pragma unroll
        for (int nt = 1; nt < kKeys / 8; ++nt) m = fmaxf(m, fmaxf(acc[mt][nt][2 * h], acc[mt][nt][2 * h + 1]));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        rm[mt][h] = m;
      }
    float mine = (c == 0) ? rm[0][0] : (c == 1) ? rm[0][1] : (c == 2) ? rm[1][0] : rm[1][1];
    run = fmaxf(run, mine);
    const int64_t key_end = (kt + 1) * kKeys;
    if (key_end % BK == 0) {  // a block is complete
      int b = (int)(key_end / BK) - 1;
      if (b < local_own) top.insert(run, b);
      run = __int_as_float(0xff800000);
    }
  }

  if (t_own < N) {
    int32_t* out = block_idx + ((int64_t)g * N + t_own) * k;
    out[0] = (int32_t)local_own;
    if (k > 1) top.emit(k - 1, out + 1);
  }
}

template <int DI, int BK, int CAP>
cudaError_t launch_t(const void* q_idx, const void* k_idx, int64_t N, int G, int k, int32_t* block_idx,
                     cudaStream_t s) {
  constexpr int LDS = DI + 8;
  const size_t smem = (size_t)(kRows + 2 * kKeys) * LDS * sizeof(uint16_t);
  auto kern = select_kernel<DI, BK, CAP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((N + kRows - 1) / kRows), (unsigned)G);
  kern<<<grid, kThreads, smem, s>>>((const uint16_t*)q_idx, (const uint16_t*)k_idx, N, G, k, block_idx);
  return cudaGetLastError();
}

template <int DI, int BK>
cudaError_t launch_cap(const void* q_idx, const void* k_idx, int64_t N, int G, int k, int32_t* block_idx,
                       cudaStream_t s) {
  int km1 = k - 1;
  if (km1 <= 4) return launch_t<DI, BK, 4>(q_idx, k_idx, N, G, k, block_idx, s);
  if (km1 <= 8) return launch_t<DI, BK, 8>(q_idx, k_idx, N, G, k, block_idx, s);
  if (km1 <= 16) return launch_t<DI, BK, 16>(q_idx, k_idx, N, G, k, block_idx, s);
  return launch_t<DI, BK, 32>(q_idx, k_idx, N, G, k, block_idx, s);
}

template <int DI>
cudaError_t launch_bk(const void* q_idx, const void* k_idx, int64_t N, int G, int Bk, int k, int32_t* block_idx,
                      cudaStream_t s) {
  if (Bk == 64) return launch_cap<DI, 64>(q_idx, k_idx, N, G, k, block_idx, s);
  return launch_cap<DI, 128>(q_idx, k_idx, N, G, k, block_idx, s);
}

}  // namespace

cudaError_t launch_select(const void* q_idx, const void* k_idx, int64_t N, int G, int d_I, int Bk, int k,
                          int32_t* block_idx, DeviceStatus* st, cudaStream_t s) {
  (void)st;
  if (d_I == 32) return launch_bk<32>(q_idx, k_idx, N, G, Bk, k, block_idx, s);
  if (d_I == 64) return launch_bk<64>(q_idx, k_idx, N, G, Bk, k, block_idx, s);
  return launch_bk<128>(q_idx, k_idx, N, G, Bk, k, block_idx, s);
}

}  // namespace msa
