// msa_invert_blocks: B -> B* (Flash-MSA "バックワードパス": the
// [head, query, slot] -> block map inverted into [head, block] -> queries;
// "MSA" study note 3-5: the reverse index that gathers, per KV block, the
// queries that chose it).
//
// A stable counting sort keyed by block id over the entries e = t*k + slot,
// which are already in ascending t:
//   1. count:   per (group, chunk of positions) a shared-memory histogram;
//   2. prefix:  per (group, block) the running sum over chunks (in place);
//   3. scan:    per group the exclusive scan over blocks -> row_ptr;
//   4. scatter: one warp per chunk walks its entries in order; lanes holding
//               the same block are ranked by lane (= entry order) with
//               __match_any_sync, so every list comes out in ascending t and
//               the result does not depend on scheduling.
#include "msa_common.cuh"

namespace msa {

namespace {

__global__ void inv_count_kernel(const int32_t* __restrict__ B, int64_t N, int k, int64_t nb, int chunk,
                                 int n_chunks, int32_t* __restrict__ counts, DeviceStatus* st) {
  extern __shared__ int32_t hist[];
  const int c = blockIdx.x, g = blockIdx.y;
  for (int64_t b = threadIdx.x; b < nb; b += blockDim.x) hist[b] = 0;
  __syncthreads();
  const int64_t e0 = (int64_t)c * chunk * k;
  const int64_t e1 = min((int64_t)(c + 1) * chunk, N) * k;
  const int32_t* Bg = B + (int64_t)g * N * k;
  for (int64_t e = e0 + threadIdx.x; e < e1; e += blockDim.x) {
    int32_t b = Bg[e];
    if (b == -1) continue;
    if (b < 0 || (int64_t)b >= nb) {
      raise_error(st, kErrBadIndex, 1u);
      continue;
    }
    atomicAdd(&hist[b], 1);
  }
  __syncthreads();
  int32_t* out = counts + ((int64_t)g * n_chunks + c) * nb;
  for (int64_t b = threadIdx.x; b < nb; b += blockDim.x) out[b] = hist[b];
}

// counts[g][c][b] <- sum over c' < c; totals into row_ptr[g][b].
__global__ void inv_prefix_kernel(int32_t* __restrict__ counts, int64_t nb, int n_chunks,
                                  int32_t* __restrict__ row_ptr) {
  const int g = blockIdx.y;
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nb) return;
  int32_t run = 0;
  int32_t* col = counts + (int64_t)g * n_chunks * nb + b;
  for (int c = 0; c < n_chunks; ++c) {
    int32_t x = col[(int64_t)c * nb];
    col[(int64_t)c * nb] = run;
    run += x;
  }
  row_ptr[(int64_t)g * (nb + 1) + b] = run;
}

// In-place exclusive scan of row_ptr[g][0..nb), row_ptr[g][nb] = total.
__global__ void __launch_bounds__(1024) inv_scan_kernel(int32_t* __restrict__ row_ptr, int64_t nb,
                                                        int32_t* __restrict__ n_entries) {
  __shared__ int32_t warp_sums[32];
  const int g = blockIdx.x;
  int32_t* rp = row_ptr + (int64_t)g * (nb + 1);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t per = (nb + blockDim.x - 1) / blockDim.x;
  const int64_t lo = min((int64_t)tid * per, nb), hi = min(lo + per, nb);
  int32_t sum = 0;
  for (int64_t i = lo; i < hi; ++i) sum += rp[i];
  // block-wide exclusive scan of the per-thread sums
  int32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
    int32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_sums[lane] = wi - w;  // exclusive prefix of warp totals
  }
  __syncthreads();
  int32_t run = warp_sums[warp] + incl - sum;
  for (int64_t i = lo; i < hi; ++i) {
    int32_t x = rp[i];
    rp[i] = run;
    run += x;
  }
  if (tid == blockDim.x - 1) {
    rp[nb] = run;
    n_entries[g] = run;
  }
}

__global__ void __launch_bounds__(32) inv_scatter_kernel(const int32_t* __restrict__ B, int64_t N, int k, int64_t nb,
                                                         int chunk, int n_chunks,
                                                         const int32_t* __restrict__ counts,
                                                         const int32_t* __restrict__ row_ptr,
                                                         int32_t* __restrict__ entries) {
  extern __shared__ int32_t cursor[];
  const int c = blockIdx.x, g = blockIdx.y, lane = threadIdx.x;
  const int32_t* rp = row_ptr + (int64_t)g * (nb + 1);
  const int32_t* cc = counts + ((int64_t)g * n_chunks + c) * nb;
  for (int64_t b = lane; b < nb; b += 32) cursor[b] = rp[b] + cc[b];
  __syncwarp();
  const int64_t e0 = (int64_t)c * chunk * k;
  const int64_t e1 = min((int64_t)(c + 1) * chunk, N) * k;
  const int32_t* Bg = B + (int64_t)g * N * k;
  int32_t* Eg = entries + (int64_t)g * N * k;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int64_t base = e0; base < e1; base += 32) {
    int64_t e = base + lane;
    int32_t b = (e < e1) ? Bg[e] : -1;
    bool valid = b >= 0 && (int64_t)b < nb;
    int key = valid ? b : -2 - lane;  // invalid lanes match nobody
    unsigned peers = __match_any_sync(0xffffffffu, key);
    int leader = __ffs(peers) - 1;
    int32_t pos = 0;
    if (valid && lane == leader) {
      pos = cursor[b];
      cursor[b] = pos + __popc(peers);
    }
    pos = __shfl_sync(0xffffffffu, pos, leader);
    if (valid) Eg[pos + __popc(peers & lt_mask)] = (int32_t)e;
    __syncwarp();
  }
}

}  // namespace

static void invert_geometry(int64_t N, int& chunk, int& n_chunks) {
  int64_t ch = (N + 255) / 256;
  if (ch < 256) ch = 256;
  ch = (ch + 31) / 32 * 32;
  chunk = (int)ch;
  n_chunks = (int)((N + ch - 1) / ch);
}

size_t invert_scratch_bytes(int64_t N, int G, int Bk, int k) {
  (void)k;
  int chunk, n_chunks;
  invert_geometry(N, chunk, n_chunks);
  int64_t nb = (N + Bk - 1) / Bk;
  return align_up((size_t)G * n_chunks * nb * sizeof(int32_t), 256);
}

InvertScratch invert_scratch_carve(void* base, int64_t N, int G, int Bk, int k) {
  (void)G;
  (void)Bk;
  (void)k;
  InvertScratch s;
  invert_geometry(N, s.chunk, s.n_chunks);
  s.counts = (int32_t*)base;
  return s;
}

cudaError_t launch_invert(const int32_t* block_idx, int64_t N, int G, int Bk, int k, int32_t* row_ptr,
                          int32_t* entries, int32_t* n_entries, const InvertScratch& sc, DeviceStatus* st,
                          cudaStream_t s) {
  const int64_t nb = (N + Bk - 1) / Bk;
  const size_t hist_bytes = (size_t)nb * sizeof(int32_t);
  cudaError_t e;
  e = cudaFuncSetAttribute(inv_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hist_bytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(inv_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hist_bytes);
  if (e != cudaSuccess) return e;
  dim3 grid_c((unsigned)sc.n_chunks, (unsigned)G);
  inv_count_kernel<<<grid_c, 256, hist_bytes, s>>>(block_idx, N, k, nb, sc.chunk, sc.n_chunks, sc.counts, st);
  dim3 grid_p((unsigned)((nb + 255) / 256), (unsigned)G);
  inv_prefix_kernel<<<grid_p, 256, 0, s>>>(sc.counts, nb, sc.n_chunks, row_ptr);
  inv_scan_kernel<<<G, 1024, 0, s>>>(row_ptr, nb, n_entries);
  inv_scatter_kernel<<<grid_c, 32, hist_bytes, s>>>(block_idx, N, k, nb, sc.chunk, sc.n_chunks, sc.counts, row_ptr,
                                                    entries);
  return cudaGetLastError();
}

}  // namespace msa
