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
//   4. scatter: one warp per chunk walks its block ids in order, staged in
//               shared memory ahead of use; lanes holding the same block are
//               ranked by lane (= entry order) with __match_any_sync, so every
//               list comes out in ascending t and the result does not depend
//               on scheduling.
#include "msa_common.cuh"

namespace msa {

namespace {

__host__ __device__ inline int64_t align_up_i(int64_t n) { return (n + 3) & ~(int64_t)3; }

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

// counts[g][c][b] <- sum over c' < c; totals into row_ptr[g][b].  A CTA takes
// 32 consecutive blocks of one group (lane = block, so every row of 32 counts
// is one coalesced 128-byte access); its 8 warps split the chunk axis into
// contiguous ranges, sum them, exchange the range totals through shared
// memory and write the running prefix in a second pass over their range.
constexpr int kPrefixWarps = 8;
__global__ void __launch_bounds__(kPrefixWarps * 32) inv_prefix_kernel(int32_t* __restrict__ counts, int64_t nb,
                                                                       int n_chunks, int32_t* __restrict__ row_ptr) {
  __shared__ int32_t wsum[kPrefixWarps][32];
  const int g = blockIdx.y, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t b = (int64_t)blockIdx.x * 32 + lane;
  const int per = (n_chunks + kPrefixWarps - 1) / kPrefixWarps;
  const int c0 = min(warp * per, n_chunks), c1 = min(c0 + per, n_chunks);
  int32_t* col = counts + (int64_t)g * n_chunks * nb + b;
  int32_t sum = 0;
  if (b < nb)
    for (int c = c0; c < c1; ++c) sum += col[(int64_t)c * nb];
  wsum[warp][lane] = sum;
  __syncthreads();
  int32_t run = 0;
  for (int w = 0; w < warp; ++w) run += wsum[w][lane];
  if (b < nb) {
    for (int c = c0; c < c1; ++c) {
      const int32_t x = col[(int64_t)c * nb];
      col[(int64_t)c * nb] = run;
      run += x;
    }
    if (warp == kPrefixWarps - 1) row_ptr[(int64_t)g * (nb + 1) + b] = run;
  }
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

// One warp per (chunk, group), so that every chunk's warp is resident at
// once.  The chunk's block ids are staged in shared memory kScatterSub at a
// time, double-buffered with cp.async (the next part lands while this one is
// ranked), so the serial ranking rounds read no global memory.
constexpr int kScatterSub = 1024;  // entries per staging buffer
__device__ __forceinline__ void cp_async_4(int32_t* smem_dst, const int32_t* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
__global__ void __launch_bounds__(32) inv_scatter_kernel(const int32_t* __restrict__ B, int64_t N, int k, int64_t nb,
                                                         int chunk, int n_chunks, const int32_t* __restrict__ counts,
                                                         const int32_t* __restrict__ row_ptr,
                                                         int32_t* __restrict__ entries) {
  extern __shared__ int32_t sc_smem[];
  int32_t* cursor = sc_smem;               // [nb]
  int32_t* sb = sc_smem + align_up_i(nb);  // [2][kScatterSub]
  const int c = blockIdx.x, g = blockIdx.y, lane = threadIdx.x;
  const int32_t* rp = row_ptr + (int64_t)g * (nb + 1);
  const int32_t* cc = counts + ((int64_t)g * n_chunks + c) * nb;
  for (int64_t b = lane; b < nb; b += 32) cursor[b] = rp[b] + cc[b];
  const int64_t e0 = (int64_t)c * chunk * k;
  const int64_t e1 = min((int64_t)(c + 1) * chunk, N) * k;
  const int32_t* Bg = B + (int64_t)g * N * k;
  int32_t* Eg = entries + (int64_t)g * N * k;
  const unsigned lt_mask = (1u << lane) - 1u;
  auto stage = [&](int64_t s0, int buf) {
    const int n = (int)min((int64_t)kScatterSub, e1 - s0);
    for (int i = lane; i < n; i += 32) cp_async_4(sb + buf * kScatterSub + i, Bg + s0 + i);
    cp_async_commit();
  };
  if (e0 < e1) stage(e0, 0);
  int buf = 0;
  for (int64_t s0 = e0; s0 < e1; s0 += kScatterSub, buf ^= 1) {
    if (s0 + kScatterSub < e1) {
      stage(s0 + kScatterSub, buf ^ 1);  // that buffer's previous part was ranked last round
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncwarp();
    const int n = (int)min((int64_t)kScatterSub, e1 - s0);
    const int32_t* ids = sb + buf * kScatterSub;
    for (int base = 0; base < n; base += 32) {
      const int i = base + lane;
      const int32_t b = i < n ? ids[i] : -1;
      const bool valid = b >= 0 && (int64_t)b < nb;
      const int key = valid ? b : -2 - lane;  // invalid lanes match nobody
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      const int leader = __ffs(peers) - 1;
      int32_t pos = 0;
      if (valid && lane == leader) {
        pos = cursor[b];
        cursor[b] = pos + __popc(peers);
      }
      pos = __shfl_sync(0xffffffffu, pos, leader);
      if (valid) Eg[pos + __popc(peers & lt_mask)] = (int32_t)(s0 + i);
      __syncwarp();
    }
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
  const size_t scatter_bytes = (size_t)(align_up_i(nb) + 2 * kScatterSub) * sizeof(int32_t);
  e = cudaFuncSetAttribute(inv_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scatter_bytes);
  if (e != cudaSuccess) return e;
  dim3 grid_c((unsigned)sc.n_chunks, (unsigned)G);
  inv_count_kernel<<<grid_c, 256, hist_bytes, s>>>(block_idx, N, k, nb, sc.chunk, sc.n_chunks, sc.counts, st);
  dim3 grid_p((unsigned)((nb + 31) / 32), (unsigned)G);
  inv_prefix_kernel<<<grid_p, kPrefixWarps * 32, 0, s>>>(sc.counts, nb, sc.n_chunks, row_ptr);
  inv_scan_kernel<<<G, 1024, 0, s>>>(row_ptr, nb, n_entries);
  inv_scatter_kernel<<<grid_c, 32, scatter_bytes, s>>>(block_idx, N, k, nb, sc.chunk, sc.n_chunks, sc.counts, row_ptr,
                                                       entries);
  return cudaGetLastError();
}

}  // namespace msa
