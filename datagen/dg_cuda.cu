/*
 * Device (CUDA) fill routines of the seeded synthetic-input generator, used to
 * fill multi-GB input buffers in place.  Bit-identical to dg_host.c (same
 * dg_core.h).  Holds none of the sparse-attention method's arithmetic.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "dg_core.h"

__global__ void dg_fill_normal_kernel(uint16_t* __restrict__ out, int64_t n, uint64_t key,
                                      int64_t first) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x * 4;
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; i < n; i += stride) {
    if (i + 4 <= n && ((reinterpret_cast<uintptr_t>(out + i) & 7) == 0)) {
      uint16_t v0 = dg_bf16_rne(dg_normal(key, (uint64_t)(first + i)));
      uint16_t v1 = dg_bf16_rne(dg_normal(key, (uint64_t)(first + i + 1)));
      uint16_t v2 = dg_bf16_rne(dg_normal(key, (uint64_t)(first + i + 2)));
      uint16_t v3 = dg_bf16_rne(dg_normal(key, (uint64_t)(first + i + 3)));
      uint2 pk;
      pk.x = (uint32_t)v0 | ((uint32_t)v1 << 16);
      pk.y = (uint32_t)v2 | ((uint32_t)v3 << 16);
      *reinterpret_cast<uint2*>(out + i) = pk;
    } else {
      for (int64_t j = i; j < n && j < i + 4; ++j)
        out[j] = dg_bf16_rne(dg_normal(key, (uint64_t)(first + j)));
    }
  }
}

__global__ void dg_q_idx_kernel(uint16_t* __restrict__ out, int64_t n_rows,
                                const int64_t* __restrict__ pos_of_row, int64_t pos_offset,
                                uint64_t noise_key, uint64_t pick_key, int G, int d_I, int Bk, int m,
                                int cap, const int32_t* __restrict__ needle_block,
                                const float* __restrict__ u, float beta) {
  int64_t total = n_rows * G;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = i / G;
    int g = (int)(i % G);
    int64_t t = pos_of_row ? pos_of_row[r] : r + pos_offset;
    dg_q_idx_row(out + i * d_I, noise_key, pick_key, r, t, g, G, d_I, Bk, m, cap, needle_block, u,
                 beta);
  }
}

extern "C" {

/* out[i] = bf16(normal(first + i)) for i < n; out is a device pointer. */
int dg_cuda_fill_normal(void* out, int64_t n, uint64_t seed, uint32_t tensor_id, int64_t first,
                        cudaStream_t stream) {
  if (n <= 0) return 0;
  int64_t blocks = (n / 4 + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  if (blocks < 1) blocks = 1;
  dg_fill_normal_kernel<<<(unsigned)blocks, 256, 0, stream>>>((uint16_t*)out, n,
                                                              dg_stream_key(seed, tensor_id), first);
  return (int)cudaGetLastError();
}

/*
 * Index-query tensor [n_rows, G, d_I] with planted needles.  Row r has query
 * position pos_of_row[r] (device array) or, when that is null, r.
 * needle_block [G*m] and u [G*m, d_I] are device arrays.
 */
int dg_cuda_q_idx(void* out, int64_t n_rows, const int64_t* pos_of_row, uint64_t seed,
                  uint32_t noise_tid, uint32_t pick_tid, int G, int d_I, int Bk, int m, int cap,
                  const int32_t* needle_block, const float* u, float beta, cudaStream_t stream) {
  if (n_rows <= 0) return 0;
  if (m > 32) return 1;
  int64_t total = n_rows * G;
  int64_t blocks = (total + 127) / 128;
  if (blocks > 152 * 64) blocks = 152 * 64;
  dg_q_idx_kernel<<<(unsigned)blocks, 128, 0, stream>>>(
      (uint16_t*)out, n_rows, pos_of_row, 0, dg_stream_key(seed, noise_tid),
      dg_stream_key(seed, pick_tid), G, d_I, Bk, m, cap, needle_block, u, beta);
  return (int)cudaGetLastError();
}

}  // extern "C"
