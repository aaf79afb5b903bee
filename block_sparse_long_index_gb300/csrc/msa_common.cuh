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

__device__ __forceinline__ uint4 ldg_stream_16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ------------------------------------------------------------------ top-k list
// Keeps the best K (<= CAP) (score, block) pairs seen so far, best = larger
// score, then smaller block id.  Slots are kept in ascending order of
// goodness: slot 0 is the worst kept pair (the eviction candidate).  Slots
// K..CAP-1 are locked with (+inf, INT_MIN), which outrank every real pair and
// stay at the top; unfilled real slots hold (-inf, INT_MAX).  All indexing is
// static so the list lives in registers.
__device__ __forceinline__ bool worse(float s1, int b1, float s2, int b2) {
  return s1 < s2 || (s1 == s2 && b1 > b2);
}

template <int CAP>
struct TopK {
  float sc[CAP];
  int ix[CAP];

  __device__ __forceinline__ void init(int K) {
#pragma unroll
    for (int i = 0; i < CAP; ++i) {
      bool locked = i >= K;
      sc[i] = locked ? __int_as_float(0x7f800000) : __int_as_float(0xff800000);
      ix[i] = locked ? INT_MIN : INT_MAX;
    }
  }

  // Cheap test for the common case: does (s, b) beat the worst kept pair?
  __device__ __forceinline__ bool admits(float s, int b) const { return worse(sc[0], ix[0], s, b); }

  __device__ __forceinline__ void insert(float s, int b) {
    if (!admits(s, b)) return;
#pragma unroll
    for (int i = 0; i < CAP; ++i) {
      float o_s = sc[i];
      int o_b = ix[i];
      if (i + 1 < CAP) {
        float n_s = sc[i + 1];
        int n_b = ix[i + 1];
        if (worse(n_s, n_b, s, b)) {  // the next pair moves down one slot
          sc[i] = n_s;
          ix[i] = n_b;
        } else if (i == 0 || worse(o_s, o_b, s, b)) {
          sc[i] = s;
          ix[i] = b;
        }
      } else if (i == 0 || worse(o_s, o_b, s, b)) {
        sc[i] = s;
        ix[i] = b;
      }
    }
  }

  // Writes the kept pairs best-first into out[0..K) (-1 where unfilled);
  // returns how many are real.
  __device__ __forceinline__ int emit(int K, int32_t* out, float* out_s = nullptr) const {
    int n = 0;
#pragma unroll
    for (int i = CAP - 1; i >= 0; --i) {
      if (ix[i] != INT_MIN && ix[i] != INT_MAX) {
        out[n] = ix[i];
        if (out_s) out_s[n] = sc[i];
        ++n;
      }
    }
    for (int i = n; i < K; ++i) out[i] = -1;
    return n;
  }
};

__host__ __device__ constexpr int topk_cap(int km1) { return km1 <= 4 ? 4 : km1 <= 8 ? 8 : km1 <= 16 ? 16 : 32; }

}  // namespace msa
