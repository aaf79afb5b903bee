// Shared device helpers of libmsa: bf16 packing, warp-level MMA and shared
// memory movement, the register-resident top-k list, the device error word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "msa_internal.h"

namespace msa {

// ------------------------------------------------------------------ errors
// The first bytes of every workspace hold a DeviceStatus; kernels raise bits
// with atomicOr and never trap.
struct DeviceStatus {
  unsigned int flags;       // kErrBadIndex | kErrTimeout
  unsigned int first_code;  // kernel-specific code of the first bad entry
  unsigned int pad[62];
};
static_assert(sizeof(DeviceStatus) == 256, "status header is 256 bytes");

constexpr unsigned int kErrBadIndex = 1u;
constexpr unsigned int kErrTimeout = 2u;

__device__ __forceinline__ void raise_error(DeviceStatus* st, unsigned int flag, unsigned int code) {
  if (st == nullptr) return;
  unsigned int old = atomicOr(&st->flags, flag);
  if (old == 0) atomicExch(&st->first_code, code);
}

__device__ __forceinline__ int64_t CacheMap::row(int64_t seq, int64_t key, DeviceStatus* st) const {
  const int64_t lp = key / page;
  int32_t pp = __ldg(table + seq * max_pages + lp);
  if (pp < 0 || (int64_t)pp >= n_pages) {
    raise_error(st, kErrBadIndex, 3u);
    pp = 0;
  }
  return (int64_t)pp * page + (key - lp * page);
}

// ------------------------------------------------------------------ bf16
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------------------ smem / async copies
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global->shared copy; src_bytes < 16 zero-fills the rest.
__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* gmem_src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem_dst)), "l"(gmem_src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                            const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                                  const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// D = A(16x32 e4m3, row) * B(32x8 e4m3, col) + D, fp32 accumulate.  Each
// fragment register holds four consecutive k of one row (A) or column (B).
__device__ __forceinline__ void mma_e4m3_16832(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Programmatic dependent launch: a primary grid lets its dependent grid be
// scheduled; the dependent waits for the primary's completion and memory.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

__device__ __forceinline__ uint4 ldg_stream_16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ------------------------------------------------------------------ top-k list
// (score, block) pairs ranked by one unsigned 64-bit key: larger key = better
// pair = larger score, then smaller block id.  The high word orders fp32
// scores as unsigned integers (-0 is first made +0, so that equal scores tie
// and fall to the block id); the low word is the complement of the id.
__device__ __forceinline__ uint64_t rank_key(float s, int32_t b) {
  uint32_t u = __float_as_uint(s + 0.0f);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((uint64_t)u << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)b);
}
__device__ __forceinline__ float rank_key_score(uint64_t key) {
  const uint32_t u = (uint32_t)(key >> 32);
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}
__device__ __forceinline__ int32_t rank_key_block(uint64_t key) {
  return (int32_t)(0xFFFFFFFFu - (uint32_t)key);
}

// Keeps the best K (<= CAP) pairs seen so far as keys in ascending order:
// slot 0 is the worst kept pair (the eviction candidate).  Slots K..CAP-1 are
// locked with the largest key and stay on top; unfilled real slots hold key 0,
// which every real pair beats.  All indexing is static so the list lives in
// registers; an insertion is one compare and two selects per slot.
template <int CAP>
struct TopK {
  uint64_t key[CAP];

  __device__ __forceinline__ void init(int K) {
#pragma unroll
    for (int i = 0; i < CAP; ++i) key[i] = i >= K ? ~0ull : 0ull;
  }

  __device__ __forceinline__ bool admits(float s, int b) const { return rank_key(s, b) > key[0]; }

  __device__ __forceinline__ void insert(float s, int b) { insert_key(rank_key(s, b)); }

  __device__ __forceinline__ void insert_key(uint64_t x) {
    if (x <= key[0]) return;
    // below[i]: slot i holds a worse pair than x (true for a prefix of the slots)
    bool below[CAP];
#pragma unroll
    for (int i = 0; i < CAP; ++i) below[i] = key[i] < x;
    // the prefix shifts down one slot and x takes the last place of the prefix
#pragma unroll
    for (int i = 0; i < CAP; ++i) {
      const bool next_below = i + 1 < CAP && below[i + 1];
      key[i] = next_below ? key[i + 1 < CAP ? i + 1 : i] : (below[i] ? x : key[i]);
    }
  }

  // Writes the kept pairs best-first into out[0..K) (-1 where unfilled);
  // returns how many are real.
  __device__ __forceinline__ int emit(int K, int32_t* out, float* out_s = nullptr) const {
    int n = 0;
#pragma unroll
    for (int i = CAP - 1; i >= 0; --i) {
      if (key[i] != 0ull && key[i] != ~0ull) {
        out[n] = rank_key_block(key[i]);
        if (out_s) out_s[n] = rank_key_score(key[i]);
        ++n;
      }
    }
    for (int i = n; i < K; ++i) out[i] = -1;
    return n;
  }
};

__host__ __device__ constexpr int topk_cap(int km1) { return km1 <= 4 ? 4 : km1 <= 8 ? 8 : km1 <= 16 ? 16 : 32; }

}  // namespace msa
