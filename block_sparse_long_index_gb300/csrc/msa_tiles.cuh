// mma.sync building blocks shared by the tile kernels that keep bf16 tiles in
// shared memory: the swizzled tile layout, ldmatrix fragment loads, paired
// m16n8k16 MMAs, accumulator-to-operand repacking, fp32 reductions to global
// memory and cp.async row loads.
#pragma once

#include "msa_common.cuh"

namespace msa {
namespace tiles {

// ------------------------------------------------------------------ shared-memory tiles
// A bf16 tile with `cols` elements per row keeps 16-byte chunk c of row r at
// chunk swz(r, c): the 8 row addresses of an ldmatrix at one chunk then fall
// in distinct banks (rows of >= 8 chunks: XOR with r mod 8; rows of 4 chunks:
// XOR with (r / 2) mod 4).
__device__ __forceinline__ int swz(int r, int c, int cpr) { return cpr >= 8 ? (c ^ (r & 7)) : (c ^ ((r >> 1) & 3)); }
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int r, int col, int cols) {
  return base + (uint32_t)(r * cols * 2 + swz(r, col >> 3, cols >> 3) * 16 + (col & 7) * 2);
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// A fragment (16 x 16) of rows r0.. and columns k0.. of a row-major tile
__device__ __forceinline__ void lds_a(uint32_t (&a)[4], uint32_t base, int r0, int k0, int cols) {
  const int lane = threadIdx.x & 31, m = lane >> 3;
  ldsm_x4(a, tile_addr(base, r0 + ((m & 1) << 3) + (lane & 7), k0 + ((m >> 1) << 3), cols));
}
// B fragments of n-tiles n0 and n0+8 (k0..k0+15) from a tile stored [n][k]
__device__ __forceinline__ void lds_b_nk(uint32_t (&b)[4], uint32_t base, int n0, int k0, int cols) {
  const int lane = threadIdx.x & 31;
  ldsm_x4(b, tile_addr(base, n0 + (lane & 7) + ((lane >> 4) << 3), k0 + (((lane >> 3) & 1) << 3), cols));
}
// B fragments of n-tiles n0 and n0+8 (k0..k0+15) from a tile stored [k][n]
__device__ __forceinline__ void lds_b_kn(uint32_t (&b)[4], uint32_t base, int k0, int n0, int cols) {
  const int lane = threadIdx.x & 31;
  ldsm_x4_t(b, tile_addr(base, k0 + (lane & 7) + (((lane >> 3) & 1) << 3), n0 + ((lane >> 4) << 3), cols));
}
__device__ __forceinline__ void mma2(float (&c0)[4], float (&c1)[4], const uint32_t (&a)[4], const uint32_t (&b)[4]) {
  const uint32_t b0[2] = {b[0], b[1]}, b1[2] = {b[2], b[3]};
  mma_bf16_16816(c0, a, b0);
  mma_bf16_16816(c1, a, b1);
}
// A fragment (16 rows x 16 k) from two m16n8 accumulator tiles (columns k 0-7 and 8-15)
__device__ __forceinline__ void c_to_a(uint32_t (&a)[4], const float (&c0)[4], const float (&c1)[4]) {
  a[0] = pack_bf16x2(c0[0], c0[1]);
  a[1] = pack_bf16x2(c0[2], c0[3]);
  a[2] = pack_bf16x2(c1[0], c1[1]);
  a[3] = pack_bf16x2(c1[2], c1[3]);
}
__device__ __forceinline__ void red_add2(float* p, float x, float y) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};\n" ::"l"(p), "f"(x), "f"(y) : "memory");
}
__device__ __forceinline__ void st_bf16(uint16_t* base, int r, int col, int cols, float v) {
  uint16_t* p = reinterpret_cast<uint16_t*>(reinterpret_cast<char*>(base) + r * cols * 2 +
                                            swz(r, col >> 3, cols >> 3) * 16 + (col & 7) * 2);
  *p = (uint16_t)(pack_bf16x2(v, 0.f) & 0xFFFFu);
}

// Rows [0, nrows) of a tile with `cols` bf16 per row: row r from src(r), or
// zeros where src(r) is null (`any` is a valid global address for those copies).
template <typename F>
__device__ __forceinline__ void load_rows(uint16_t* dst, int nrows, int cols, const uint16_t* any, F src) {
  const int cpr = cols >> 3;
  for (int i = threadIdx.x; i < nrows * cpr; i += blockDim.x) {
    const int r = i / cpr, c = i % cpr;
    const uint16_t* gp = src(r);
    cp_async_16(reinterpret_cast<char*>(dst) + r * cols * 2 + swz(r, c, cpr) * 16, gp ? gp + c * 8 : any,
                gp ? 16 : 0);
  }
}

}  // namespace tiles
}  // namespace msa
