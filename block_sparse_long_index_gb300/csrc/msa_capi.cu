// C ABI of libmsa.so: argument validation, workspace sizing and layout,
// device error word, dispatch to the kernel translation units.
// The declarations and their contracts are in include/msa.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "../../include/msa.h"
#include "msa_common.cuh"

namespace msa {

int num_sms() {
  static int cached_dev = -1;
  static int cached = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev != cached_dev) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached = n;
    cached_dev = dev;
  }
  return cached;
}

static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return nullptr;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return encode;
}

static CUtensorMapSwizzle swizzle_of(int swizzle_bytes) {
  return swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
         : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
         : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                               : CU_TENSOR_MAP_SWIZZLE_NONE;
}

bool encode_tmap_2d(void* tmap, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride_bytes,
                    uint32_t box_inner, uint32_t box_rows, int swizzle_bytes, int elem_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (!encode) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = encode(reinterpret_cast<CUtensorMap*>(tmap), dt, 2,
                      const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      swizzle_of(swizzle_bytes), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_3d(void* tmap, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
                    uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2, int swizzle_bytes, int elem_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (!encode) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = encode(reinterpret_cast<CUtensorMap*>(tmap), dt, 3,
                      const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      swizzle_of(swizzle_bytes), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_4d(void* tmap, const void* base, const uint64_t dims[4], const uint64_t strides_bytes[3],
                    const uint32_t box[4], int swizzle_bytes) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (!encode) return false;
  cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t s[3] = {strides_bytes[0], strides_bytes[1], strides_bytes[2]};
  cuuint32_t b[4] = {box[0], box[1], box[2], box[3]};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(reinterpret_cast<CUtensorMap*>(tmap), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                      const_cast<void*>(base), d, s, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_of(swizzle_bytes),
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace msa

using msa::align_up;

namespace {

constexpr size_t kHeader = sizeof(msa::DeviceStatus);  // 256 bytes at the start of every workspace

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2_upto8(int x) { return x == 1 || x == 2 || x == 4 || x == 8; }

msa_status_t check_common(int64_t N, int G, int d_I, int Bk, int k) {
  if (N < 1 || G < 1 || d_I < 1 || Bk < 1 || k < 1) return MSA_ERR_INVALID_ARGUMENT;
  if (G > 64 || (d_I != 32 && d_I != 64 && d_I != 128) || (Bk != 64 && Bk != 128) || k > 32)
    return MSA_ERR_UNSUPPORTED;
  const int64_t nb = (N + Bk - 1) / Bk;
  if (nb > 32768 || N * (int64_t)k >= ((int64_t)1 << 31)) return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

msa_status_t check_shape(const msa_shape_t* s) {
  if (!s) return MSA_ERR_INVALID_ARGUMENT;
  if (s->H_q < 1 || s->H_kv < 1 || s->d < 1) return MSA_ERR_INVALID_ARGUMENT;
  if (s->H_q % s->H_kv != 0) return MSA_ERR_INVALID_ARGUMENT;
  msa_status_t st = check_common(s->N, s->H_kv, s->d_I, s->Bk, s->k);
  if (st != MSA_OK) return st;
  if (!pow2_upto8(s->H_q / s->H_kv) || (s->d != 64 && s->d != 128)) return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

// Validates the workspace and clears its first `clear` bytes (the status header
// and, for calls that keep completion counters there, those counters).
msa_status_t begin(void* ws, size_t ws_bytes, size_t need, cudaStream_t s, size_t clear = kHeader) {
  if (!ws) return MSA_ERR_INVALID_ARGUMENT;
  if (((uintptr_t)ws & 255u) != 0) return MSA_ERR_INVALID_ARGUMENT;
  if (ws_bytes < need) return MSA_ERR_WORKSPACE_TOO_SMALL;
  if (cudaMemsetAsync(ws, 0, clear, s) != cudaSuccess) return MSA_ERR_CUDA;
  return MSA_OK;
}

msa_status_t finish(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA; }

}  // namespace

extern "C" {

size_t msa_select_blocks_workspace(int64_t N, int G, int d_I, int Bk, int k) {
  (void)N;
  (void)G;
  (void)d_I;
  (void)Bk;
  (void)k;
  return kHeader;
}

static msa_status_t select_impl(const void* q_idx, const void* k_idx, int64_t N, int G, int d_I, int Bk, int k,
                                int32_t* block_idx, void* workspace, size_t workspace_bytes, msa_stream_t stream,
                                bool f8) {
  if (!q_idx || !k_idx || !block_idx) return MSA_ERR_INVALID_ARGUMENT;
  msa_status_t st = check_common(N, G, d_I, Bk, k);
  if (st != MSA_OK) return st;
  if (f8 && d_I == 32) return MSA_ERR_UNSUPPORTED;
  if (!aligned16(q_idx) || !aligned16(k_idx) || ((uintptr_t)block_idx & 3u)) return MSA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = (cudaStream_t)stream;
  st = begin(workspace, workspace_bytes, msa_select_blocks_workspace(N, G, d_I, Bk, k), s);
  if (st != MSA_OK) return st;
  return finish(
      msa::launch_select(q_idx, k_idx, N, G, d_I, Bk, k, block_idx, (msa::DeviceStatus*)workspace, s, f8));
}

msa_status_t msa_select_blocks(const void* q_idx, const void* k_idx, int64_t N, int G, int d_I, int Bk, int k,
                               int32_t* block_idx, void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  return select_impl(q_idx, k_idx, N, G, d_I, Bk, k, block_idx, workspace, workspace_bytes, stream, false);
}

msa_status_t msa_select_blocks_fp8(const void* q_idx, const void* k_idx, int64_t N, int G, int d_I, int Bk, int k,
                                   int32_t* block_idx, void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  return select_impl(q_idx, k_idx, N, G, d_I, Bk, k, block_idx, workspace, workspace_bytes, stream, true);
}

size_t msa_select_blocks_varlen_workspace(int64_t N, int G, int d_I, int Bk, int k) {
  (void)G;
  (void)d_I;
  (void)k;
  if (N < 1 || Bk < 1) return kHeader;
  return kHeader + msa::align_up((size_t)((N + Bk - 1) / Bk) * 4, 256);
}

msa_status_t msa_select_blocks_varlen(const void* q_idx, const void* k_idx, const int32_t* cu_seqlens, int S,
                                      int64_t N, int G, int d_I, int Bk, int k, int32_t* block_idx, void* workspace,
                                      size_t workspace_bytes, msa_stream_t stream) {
  if (!q_idx || !k_idx || !block_idx || !cu_seqlens || S < 1) return MSA_ERR_INVALID_ARGUMENT;
  msa_status_t st = check_common(N, G, d_I, Bk, k);
  if (st != MSA_OK) return st;
  if (!aligned16(q_idx) || !aligned16(k_idx) || ((uintptr_t)block_idx & 3u) || ((uintptr_t)cu_seqlens & 3u))
    return MSA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = (cudaStream_t)stream;
  st = begin(workspace, workspace_bytes, msa_select_blocks_varlen_workspace(N, G, d_I, Bk, k), s);
  if (st != MSA_OK) return st;
  int32_t* blk_lo = (int32_t*)((char*)workspace + kHeader);
  msa::DeviceStatus* dst = (msa::DeviceStatus*)workspace;
  cudaError_t e = msa::launch_varlen_blocks(cu_seqlens, S, N, Bk, blk_lo, dst, s);
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  return finish(msa::launch_select(q_idx, k_idx, N, G, d_I, Bk, k, block_idx, dst, s, false, blk_lo));
}

msa_status_t msa_quantize_e4m3(const void* x, int64_t n, float scale, void* y, msa_stream_t stream) {
  if (n < 0 || ((!x || !y) && n > 0)) return MSA_ERR_INVALID_ARGUMENT;
  if (((uintptr_t)x & 1u) || scale != scale) return MSA_ERR_INVALID_ARGUMENT;
  return finish(msa::launch_quantize_e4m3(x, n, scale, y, (cudaStream_t)stream));
}

size_t msa_invert_blocks_workspace(int64_t N, int G, int Bk, int k) {
  if (N < 1 || G < 1 || Bk < 1 || k < 1) return kHeader;
  return kHeader + msa::invert_scratch_bytes(N, G, Bk, k);
}

msa_status_t msa_invert_blocks(const int32_t* block_idx, int64_t N, int G, int Bk, int k, int32_t* row_ptr,
                               int32_t* entries, int32_t* n_entries, void* workspace, size_t workspace_bytes,
                               msa_stream_t stream) {
  if (!block_idx || !row_ptr || !entries || !n_entries) return MSA_ERR_INVALID_ARGUMENT;
  msa_status_t st = check_common(N, G, 32, Bk, k);
  if (st != MSA_OK) return st;
  if (((uintptr_t)block_idx | (uintptr_t)row_ptr | (uintptr_t)entries | (uintptr_t)n_entries) & 3u)
    return MSA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = (cudaStream_t)stream;
  st = begin(workspace, workspace_bytes, msa_invert_blocks_workspace(N, G, Bk, k), s);
  if (st != MSA_OK) return st;
  msa::InvertScratch sc = msa::invert_scratch_carve((char*)workspace + kHeader, N, G, Bk, k);
  return finish(msa::launch_invert(block_idx, N, G, Bk, k, row_ptr, entries, n_entries, sc,
                                   (msa::DeviceStatus*)workspace, s));
}

size_t msa_sparse_attn_fwd_workspace(const msa_shape_t* shape) {
  if (check_shape(shape) != MSA_OK) return kHeader;
  msa::AttnPlan p = msa::attn_plan(shape->N, shape->H_q, shape->H_kv, shape->d, shape->Bk, shape->k);
  return kHeader + msa::attn_scratch_bytes(p);
}

msa_status_t msa_sparse_attn_fwd(const void* q, const void* k, const void* v, const int32_t* block_idx,
                                 const msa_shape_t* shape, float scale, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, msa_stream_t stream) {
  if (!q || !k || !v || !block_idx || !out || !lse) return MSA_ERR_INVALID_ARGUMENT;
  msa_status_t st = check_shape(shape);
  if (st != MSA_OK) return st;
  if (!(scale > 0.f) || scale != scale) return MSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || ((uintptr_t)block_idx & 3u) ||
      ((uintptr_t)lse & 3u))
    return MSA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = (cudaStream_t)stream;
  st = begin(workspace, workspace_bytes, msa_sparse_attn_fwd_workspace(shape), s);
  if (st != MSA_OK) return st;
  msa::AttnPlan p = msa::attn_plan(shape->N, shape->H_q, shape->H_kv, shape->d, shape->Bk, shape->k);
  return finish(msa::launch_attn(q, k, v, block_idx, p, scale, out, lse, (char*)workspace + kHeader,
                                 (msa::DeviceStatus*)workspace, s));
}

size_t msa_prefill_workspace(const msa_shape_t* shape) {
  if (check_shape(shape) != MSA_OK) return kHeader;
  msa::AttnPlan p = msa::attn_plan(shape->N, shape->H_q, shape->H_kv, shape->d, shape->Bk, shape->k);
  return kHeader + msa::attn_scratch_bytes(p);
}

static msa_status_t prefill_impl(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                                 const msa_shape_t* shape, float scale, int32_t* block_idx, void* out, float* lse,
                                 void* workspace, size_t workspace_bytes, msa_stream_t stream, bool f8) {
  if (!q || !k || !v || !q_idx || !k_idx || !block_idx || !out || !lse) return MSA_ERR_INVALID_ARGUMENT;
  msa_status_t st = check_shape(shape);
  if (st != MSA_OK) return st;
  if (f8 && shape->d_I == 32) return MSA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || scale != scale) return MSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_idx) || !aligned16(k_idx) ||
      !aligned16(out) || ((uintptr_t)block_idx & 3u) || ((uintptr_t)lse & 3u))
    return MSA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = (cudaStream_t)stream;
  st = begin(workspace, workspace_bytes, msa_prefill_workspace(shape), s);
  if (st != MSA_OK) return st;
  msa::AttnPlan p = msa::attn_plan(shape->N, shape->H_q, shape->H_kv, shape->d, shape->Bk, shape->k);
  return finish(msa::launch_prefill(q, k, v, q_idx, k_idx, shape->d_I, p, scale, block_idx, out, lse,
                                    (char*)workspace + kHeader, (msa::DeviceStatus*)workspace, s, f8));
}

msa_status_t msa_prefill(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                         const msa_shape_t* shape, float scale, int32_t* block_idx, void* out, float* lse,
                         void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  return prefill_impl(q, k, v, q_idx, k_idx, shape, scale, block_idx, out, lse, workspace, workspace_bytes, stream,
                      false);
}

size_t msa_prefill_varlen_workspace(const msa_shape_t* shape) {
  if (check_shape(shape) != MSA_OK) return kHeader;
  const size_t lo_bytes = msa::align_up((size_t)((shape->N + shape->Bk - 1) / shape->Bk) * 4, 256);
  const size_t attn = msa_prefill_workspace(shape) - kHeader;
  return kHeader + (lo_bytes > attn ? lo_bytes : attn);
}

msa_status_t msa_prefill_varlen(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                                const int32_t* cu_seqlens, int S, const msa_shape_t* shape, float scale,
                                int32_t* block_idx, void* out, float* lse, void* workspace, size_t workspace_bytes,
                                msa_stream_t stream) {
  if (!q || !k || !v || !q_idx || !k_idx || !block_idx || !out || !lse || !cu_seqlens || S < 1)
    return MSA_ERR_INVALID_ARGUMENT;
  msa_status_t st = check_shape(shape);
  if (st != MSA_OK) return st;
  if (!(scale > 0.f) || scale != scale) return MSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_idx) || !aligned16(k_idx) ||
      !aligned16(out) || ((uintptr_t)block_idx & 3u) || ((uintptr_t)lse & 3u) || ((uintptr_t)cu_seqlens & 3u))
    return MSA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = (cudaStream_t)stream;
  st = begin(workspace, workspace_bytes, msa_prefill_varlen_workspace(shape), s);
  if (st != MSA_OK) return st;
  // the block map lives where the attention scratch goes later: the select has read it by then
  int32_t* blk_lo = (int32_t*)((char*)workspace + kHeader);
  msa::DeviceStatus* dst = (msa::DeviceStatus*)workspace;
  if (msa::launch_varlen_blocks(cu_seqlens, S, shape->N, shape->Bk, blk_lo, dst, s) != cudaSuccess)
    return MSA_ERR_CUDA;
  msa::AttnPlan p = msa::attn_plan(shape->N, shape->H_q, shape->H_kv, shape->d, shape->Bk, shape->k);
  return finish(msa::launch_prefill(q, k, v, q_idx, k_idx, shape->d_I, p, scale, block_idx, out, lse,
                                    (char*)workspace + kHeader, dst, s, false, blk_lo));
}

msa_status_t msa_prefill_fp8(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                             const msa_shape_t* shape, float scale, int32_t* block_idx, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, msa_stream_t stream) {
  return prefill_impl(q, k, v, q_idx, k_idx, shape, scale, block_idx, out, lse, workspace, workspace_bytes, stream,
                      true);
}

size_t msa_sparse_attn_bwd_workspace(const msa_shape_t* shape) {
  if (check_shape(shape) != MSA_OK) return kHeader;
  return kHeader + msa::bwd_scratch_bytes(shape->N, shape->H_q, shape->H_kv, shape->d, shape->Bk, shape->k);
}

msa_status_t msa_sparse_attn_bwd(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                                 const int32_t* block_idx, const void* out, const float* lse, const void* dout,
                                 const msa_shape_t* shape, float scale, float kl_weight, float* dq, float* dk,
                                 float* dv, float* dq_idx, float* dk_idx, float* kl, void* workspace,
                                 size_t workspace_bytes, msa_stream_t stream) {
  if (!q || !k || !v || !q_idx || !k_idx || !block_idx || !out || !lse || !dout || !dq || !dk || !dv || !dq_idx ||
      !dk_idx)
    return MSA_ERR_INVALID_ARGUMENT;
  msa_status_t st = check_shape(shape);
  if (st != MSA_OK) return st;
  if (!(scale > 0.f) || scale != scale || kl_weight != kl_weight) return MSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_idx) || !aligned16(k_idx) || !aligned16(out) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(dq_idx) ||
      !aligned16(dk_idx) || ((uintptr_t)block_idx & 3u) || ((uintptr_t)lse & 3u) || ((uintptr_t)kl & 3u))
    return MSA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = (cudaStream_t)stream;
  st = begin(workspace, workspace_bytes, msa_sparse_attn_bwd_workspace(shape), s);
  if (st != MSA_OK) return st;
  return finish(msa::launch_bwd(q, k, v, q_idx, k_idx, block_idx, out, lse, dout, shape->N, shape->H_q, shape->H_kv,
                                shape->d, shape->d_I, shape->Bk, shape->k, scale, kl_weight, dq, dk, dv, dq_idx,
                                dk_idx, kl, (char*)workspace + kHeader, (msa::DeviceStatus*)workspace, s));
}

static msa_status_t check_warmup(const msa_shape_t* shape, float scale) {
  msa_status_t st = check_shape(shape);
  if (st != MSA_OK) return st;
  if (!(scale > 0.f) || scale != scale) return MSA_ERR_INVALID_ARGUMENT;
  if (shape->N > ((int64_t)1 << 31) / 16 * 16) return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

msa_status_t msa_warmup_fwd(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                            const msa_shape_t* shape, float scale, void* out, float* lse, float* lse_idx,
                            msa_stream_t stream) {
  if (!q || !k || !v || !q_idx || !k_idx || !out || !lse || !lse_idx) return MSA_ERR_INVALID_ARGUMENT;
  msa_status_t st = check_warmup(shape, scale);
  if (st != MSA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_idx) || !aligned16(k_idx) || !aligned16(out) ||
      ((uintptr_t)lse & 3u) || ((uintptr_t)lse_idx & 3u))
    return MSA_ERR_INVALID_ARGUMENT;
  return finish(msa::launch_warmup(q, k, v, q_idx, k_idx, shape->N, shape->H_q, shape->H_kv, shape->d, shape->d_I,
                                   scale, 0.f, true, false, out, lse, lse_idx, nullptr, nullptr, nullptr,
                                   (cudaStream_t)stream));
}

msa_status_t msa_warmup_index_grad(const void* q, const void* k, const void* q_idx, const void* k_idx,
                                   const float* lse, const float* lse_idx, const msa_shape_t* shape, float scale,
                                   float kl_weight, float* dq_idx, float* dk_idx, float* kl, msa_stream_t stream) {
  if (!q || !k || !q_idx || !k_idx || !lse || !lse_idx || !dq_idx || !dk_idx || !kl) return MSA_ERR_INVALID_ARGUMENT;
  msa_status_t st = check_warmup(shape, scale);
  if (st != MSA_OK) return st;
  if (kl_weight != kl_weight) return MSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k) || !aligned16(q_idx) || !aligned16(k_idx) || !aligned16(dq_idx) ||
      !aligned16(dk_idx) || ((uintptr_t)lse & 3u) || ((uintptr_t)lse_idx & 3u) || ((uintptr_t)kl & 3u))
    return MSA_ERR_INVALID_ARGUMENT;
  return finish(msa::launch_warmup(q, k, nullptr, q_idx, k_idx, shape->N, shape->H_q, shape->H_kv, shape->d,
                                   shape->d_I, scale, kl_weight, false, true, nullptr, const_cast<float*>(lse),
                                   const_cast<float*>(lse_idx), dq_idx, dk_idx, kl, (cudaStream_t)stream));
}

size_t msa_decode_workspace(int B, const msa_shape_t* shape) {
  if (B < 1 || check_shape(shape) != MSA_OK) return kHeader;
  msa::DecodePlan p = msa::decode_plan(B, shape->N, shape->H_q, shape->H_kv, shape->d, shape->d_I, shape->Bk,
                                       shape->k);
  return kHeader + msa::decode_scratch_bytes(p);
}

static msa_status_t decode_impl(const void* q_t, const void* q_idx_t, const void* k_idx_cache, const void* k_cache,
                                const void* v_cache, const int32_t* ctx_len, int B, const msa_shape_t* shape,
                                float scale, void* out, float* lse, int32_t* block_idx, void* workspace,
                                size_t workspace_bytes, msa_stream_t stream, bool f8) {
  if (!q_t || !q_idx_t || !k_idx_cache || !k_cache || !v_cache || !ctx_len || !out) return MSA_ERR_INVALID_ARGUMENT;
  if (B < 1) return MSA_ERR_INVALID_ARGUMENT;
  msa_status_t st = check_shape(shape);
  if (st != MSA_OK) return st;
  if (f8 && shape->d_I == 32) return MSA_ERR_UNSUPPORTED;
  if (shape->H_kv > 8) return MSA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || scale != scale) return MSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q_t) || !aligned16(q_idx_t) || !aligned16(k_idx_cache) || !aligned16(k_cache) ||
      !aligned16(v_cache) || ((uintptr_t)ctx_len & 3u) || ((uintptr_t)out & 1u) || ((uintptr_t)lse & 3u) ||
      ((uintptr_t)block_idx & 3u))
    return MSA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = (cudaStream_t)stream;
  msa::DecodePlan p = msa::decode_plan(B, shape->N, shape->H_q, shape->H_kv, shape->d, shape->d_I, shape->Bk,
                                       shape->k);
  p.f8 = f8;
  st = begin(workspace, workspace_bytes, msa_decode_workspace(B, shape), s, kHeader + msa::decode_clear_bytes(p));
  if (st != MSA_OK) return st;
  return finish(msa::launch_decode(q_t, q_idx_t, k_idx_cache, k_cache, v_cache, ctx_len, p, scale, out, lse,
                                   block_idx, (char*)workspace + kHeader, (msa::DeviceStatus*)workspace, s));
}

msa_status_t msa_decode(const void* q_t, const void* q_idx_t, const void* k_idx_cache, const void* k_cache,
                        const void* v_cache, const int32_t* ctx_len, int B, const msa_shape_t* shape, float scale,
                        void* out, float* lse, int32_t* block_idx, void* workspace, size_t workspace_bytes,
                        msa_stream_t stream) {
  return decode_impl(q_t, q_idx_t, k_idx_cache, k_cache, v_cache, ctx_len, B, shape, scale, out, lse, block_idx,
                     workspace, workspace_bytes, stream, false);
}

msa_status_t msa_decode_fp8(const void* q_t, const void* q_idx_t, const void* k_idx_cache, const void* k_cache,
                            const void* v_cache, const int32_t* ctx_len, int B, const msa_shape_t* shape, float scale,
                            void* out, float* lse, int32_t* block_idx, void* workspace, size_t workspace_bytes,
                            msa_stream_t stream) {
  return decode_impl(q_t, q_idx_t, k_idx_cache, k_cache, v_cache, ctx_len, B, shape, scale, out, lse, block_idx,
                     workspace, workspace_bytes, stream, true);
}

static msa_status_t decode_paged_impl(const void* q_t, const void* q_idx_t, const void* k_idx_pool,
                                      const void* k_pool, const void* v_pool, const int32_t* page_table,
                                      int64_t max_pages, int64_t n_pages, int page_size, const int32_t* ctx_len, int B,
                                      const msa_shape_t* shape, float scale, void* out, float* lse,
                                      int32_t* block_idx, void* workspace, size_t workspace_bytes,
                                      msa_stream_t stream, bool f8) {
  if (!q_t || !q_idx_t || !k_idx_pool || !k_pool || !v_pool || !page_table || !ctx_len || !out)
    return MSA_ERR_INVALID_ARGUMENT;
  if (B < 1 || max_pages < 1 || n_pages < 1 || page_size < 16 || page_size % 16 != 0) return MSA_ERR_INVALID_ARGUMENT;
  msa_status_t st = check_shape(shape);
  if (st != MSA_OK) return st;
  if (shape->N != max_pages * (int64_t)page_size) return MSA_ERR_INVALID_ARGUMENT;  // capacity of a sequence
  if (f8 && shape->d_I == 32) return MSA_ERR_UNSUPPORTED;
  if (shape->H_kv > 8) return MSA_ERR_UNSUPPORTED;
  if (n_pages > (int64_t)1 << 31) return MSA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || scale != scale) return MSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q_t) || !aligned16(q_idx_t) || !aligned16(k_idx_pool) || !aligned16(k_pool) || !aligned16(v_pool) ||
      ((uintptr_t)page_table & 3u) || ((uintptr_t)ctx_len & 3u) || ((uintptr_t)out & 1u) || ((uintptr_t)lse & 3u) ||
      ((uintptr_t)block_idx & 3u))
    return MSA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = (cudaStream_t)stream;
  msa::DecodePlan p = msa::decode_plan(B, shape->N, shape->H_q, shape->H_kv, shape->d, shape->d_I, shape->Bk,
                                       shape->k);
  st = begin(workspace, workspace_bytes, msa_decode_workspace(B, shape), s, kHeader + msa::decode_clear_bytes(p));
  if (st != MSA_OK) return st;
  p.f8 = f8;
  msa::CacheMap map;
  map.table = page_table;
  map.max_pages = max_pages;
  map.n_pages = n_pages;
  map.page = page_size;
  return finish(msa::launch_decode(q_t, q_idx_t, k_idx_pool, k_pool, v_pool, ctx_len, p, scale, out, lse, block_idx,
                                   (char*)workspace + kHeader, (msa::DeviceStatus*)workspace, s, &map));
}

msa_status_t msa_decode_paged(const void* q_t, const void* q_idx_t, const void* k_idx_pool, const void* k_pool,
                              const void* v_pool, const int32_t* page_table, int64_t max_pages, int64_t n_pages,
                              int page_size, const int32_t* ctx_len, int B, const msa_shape_t* shape, float scale,
                              void* out, float* lse, int32_t* block_idx, void* workspace, size_t workspace_bytes,
                              msa_stream_t stream) {
  return decode_paged_impl(q_t, q_idx_t, k_idx_pool, k_pool, v_pool, page_table, max_pages, n_pages, page_size,
                           ctx_len, B, shape, scale, out, lse, block_idx, workspace, workspace_bytes, stream, false);
}

msa_status_t msa_decode_paged_fp8(const void* q_t, const void* q_idx_t, const void* k_idx_pool, const void* k_pool,
                                  const void* v_pool, const int32_t* page_table, int64_t max_pages, int64_t n_pages,
                                  int page_size, const int32_t* ctx_len, int B, const msa_shape_t* shape, float scale,
                                  void* out, float* lse, int32_t* block_idx, void* workspace, size_t workspace_bytes,
                                  msa_stream_t stream) {
  return decode_paged_impl(q_t, q_idx_t, k_idx_pool, k_pool, v_pool, page_table, max_pages, n_pages, page_size,
                           ctx_len, B, shape, scale, out, lse, block_idx, workspace, workspace_bytes, stream, true);
}

// The decode step without a caller workspace: its scratch is the library's
// fixed device array (see msa_decode.cu), so this call allocates nothing.
msa_status_t msa_decode_noalloc(const void* q_t, const void* q_idx_t, const void* k_idx_cache, const void* k_cache,
                                const void* v_cache, const int32_t* ctx_len, int B, const msa_shape_t* shape,
                                float scale, void* out, float* lse, int32_t* block_idx, msa_stream_t stream) {
  if (!q_t || !q_idx_t || !k_idx_cache || !k_cache || !v_cache || !ctx_len || !out) return MSA_ERR_INVALID_ARGUMENT;
  if (B < 1) return MSA_ERR_INVALID_ARGUMENT;
  msa_status_t st = check_shape(shape);
  if (st != MSA_OK) return st;
  if (shape->H_kv > 8) return MSA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || scale != scale) return MSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q_t) || !aligned16(q_idx_t) || !aligned16(k_idx_cache) || !aligned16(k_cache) ||
      !aligned16(v_cache) || ((uintptr_t)ctx_len & 3u) || ((uintptr_t)out & 1u) || ((uintptr_t)lse & 3u) ||
      ((uintptr_t)block_idx & 3u))
    return MSA_ERR_INVALID_ARGUMENT;
  const msa::DecodePlan p = msa::decode_plan(B, shape->N, shape->H_q, shape->H_kv, shape->d, shape->d_I, shape->Bk,
                                             shape->k);
  const size_t need = kHeader + msa::decode_scratch_bytes(p);
  if (need > msa::kNoAllocScratchBytes) return MSA_ERR_WORKSPACE_TOO_SMALL;  // beyond the fixed array
  void* scratch = nullptr;
  if (msa::noalloc_scratch(need, &scratch) != cudaSuccess || !scratch) return MSA_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  // the status word and the completion counters start clear
  if (cudaMemsetAsync(scratch, 0, kHeader + msa::decode_clear_bytes(p), s) != cudaSuccess) return MSA_ERR_CUDA;
  return finish(msa::launch_decode(q_t, q_idx_t, k_idx_cache, k_cache, v_cache, ctx_len, p, scale, out, lse,
                                   block_idx, (char*)scratch + kHeader, (msa::DeviceStatus*)scratch, s));
}

msa_status_t msa_check_device_error(void* workspace, msa_stream_t stream) {
  if (!workspace) return MSA_ERR_INVALID_ARGUMENT;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MSA_ERR_CUDA;
  unsigned int flags = 0;
  if (cudaMemcpy(&flags, workspace, sizeof(flags), cudaMemcpyDeviceToHost) != cudaSuccess) return MSA_ERR_CUDA;
  if (flags & msa::kErrBadIndex) return MSA_ERR_BAD_INDEX;
  if (flags & msa::kErrTimeout) return MSA_ERR_TIMEOUT;
  return MSA_OK;
}

const char* msa_status_string(msa_status_t status) {
  switch (status) {
    case MSA_OK: return "ok";
    case MSA_ERR_INVALID_ARGUMENT: return "invalid argument (null or misaligned pointer, bad size or shape)";
    case MSA_ERR_UNSUPPORTED: return "unsupported shape (see include/msa.h for the supported set)";
    case MSA_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than the *_workspace() size";
    case MSA_ERR_CUDA: return "CUDA launch or runtime error";
    case MSA_ERR_BAD_INDEX: return "bad index found on the device (entry skipped)";
    case MSA_ERR_TIMEOUT: return "a bounded device wait gave up";
    default: return "unknown status";
  }
}

}  // extern "C"
