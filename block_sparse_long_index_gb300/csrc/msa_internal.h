// Internal launch interface between the C-ABI layer (msa_capi.cu) and the
// kernel translation units.  Not part of the public header.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace msa {

struct DeviceStatus;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int num_sms();  // cached cudaDevAttrMultiProcessorCount of the current device

// 2-D tiled TMA descriptor over a row-major matrix [rows, inner] of bf16
// (elem_bytes 2) or bytes (elem_bytes 1, e.g. FP8 codes) with the given row
// stride, box {box_inner, box_rows} and swizzle (0, 32, 64 or 128 bytes);
// out-of-bounds elements read as zero.  False if the driver refuses.
bool encode_tmap_2d(void* tmap /* CUtensorMap */, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, int swizzle_bytes,
                    int elem_bytes = 2);
// 3-D variant: dims {d0, d1, d2} (d0 contiguous), byte strides of dims 1 and 2, box {b0, b1, b2}; elements
// are bf16 (elem_bytes 2) or fp32 (elem_bytes 4).
bool encode_tmap_3d(void* tmap, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1_bytes,
                    uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2, int swizzle_bytes,
                    int elem_bytes = 2);
// 4-D variant: byte strides of dims 1..3 in any order (a permuted view is allowed).
bool encode_tmap_4d(void* tmap, const void* base, const uint64_t dims[4], const uint64_t strides_bytes[3],
                    const uint32_t box[4], int swizzle_bytes);

// ---- select (msa_select.cu)
// f8: q_idx and k_idx hold FP8 E4M3 codes (d_I of 64 or 128) instead of bf16.
// blk_lo (nullable): first block of each block's sequence when several
// sequences share the cells; candidates of row t are then [blk_lo[t/Bk], t/Bk).
cudaError_t launch_select(const void* q_idx, const void* k_idx, int64_t N, int G, int d_I, int Bk, int k,
                          int32_t* block_idx, DeviceStatus* st, cudaStream_t s, bool f8 = false,
                          const int32_t* blk_lo = nullptr);
// blk_lo[nb] from the block-aligned sequence offsets cu_seqlens[S+1] (device).
cudaError_t launch_varlen_blocks(const int32_t* cu_seqlens, int S, int64_t N, int Bk, int32_t* blk_lo,
                                 DeviceStatus* st, cudaStream_t s);
// y[i] = E4M3 code of (bf16 x[i]) * scale (round to nearest even, saturated at 448).
cudaError_t launch_quantize_e4m3(const void* x, int64_t n, float scale, void* y, cudaStream_t s);

// ---- invert (msa_invert.cu)
struct InvertScratch {
  int32_t* counts;  // [G, n_chunks, nb]
  int chunk;        // positions per chunk
  int n_chunks;
};
size_t invert_scratch_bytes(int64_t N, int G, int Bk, int k);
InvertScratch invert_scratch_carve(void* base, int64_t N, int G, int Bk, int k);
cudaError_t launch_invert(const int32_t* block_idx, int64_t N, int G, int Bk, int k, int32_t* row_ptr,
                          int32_t* entries, int32_t* n_entries, const InvertScratch& sc, DeviceStatus* st,
                          cudaStream_t s);

// ---- attention (msa_attn.cu)
// One record of a slab's flat work list: (group g, block b) and up to
// kTilePositions query positions that chose b, with each position's slot in
// its block set.  Written by the schedule, copied whole into shared memory by
// the tile kernels (128 bytes, 16-byte aligned).  A tile of the forward
// attention is ppr consecutive records of one (g, b) (16 ppr positions x gs
// heads = 128 MMA rows, ppr = 8 / gs); a record past the tile's last position
// has count 0 and every t = -1.
constexpr int kTilePositions = 16;
struct alignas(16) TileRecord {
  int32_t gb;     // g * nb + b
  int32_t g, b;
  int32_t count;  // positions in the tile, 1..16
  int32_t t[kTilePositions];
  uint8_t slot[kTilePositions];
  int32_t pad[4 + 4];
};
static_assert(sizeof(TileRecord) == 128, "tile record is one 128-byte line");

struct AttnPlan {
  int64_t N;
  int H_q, H_kv, d, Bk, k, gs;
  int ppr;            // records (of 16 positions) per tile: 8 / gs
  int64_t nb;
  int64_t slab;       // query positions per slab
  int64_t max_tiles;  // bound on the tiles of one slab (each ppr records)
};
AttnPlan attn_plan(int64_t N, int H_q, int H_kv, int d, int Bk, int k);
size_t attn_scratch_bytes(const AttnPlan& p);
// The tcgen05 tile kernel of one query slab (msa_attn_tile.cu).
cudaError_t launch_attn_tiles(const void* q, const void* k, const void* v, const TileRecord* rec,
                              const int32_t* tile_off, int64_t N, int H_q, int H_kv, int d, int Bk, int k_blocks,
                              int64_t nb, int gs, int ppr, int64_t T0, int64_t T1, int64_t rows, int64_t max_tiles,
                              float scale,
                              uint16_t* part_o, float2* part_ml, DeviceStatus* st, cudaStream_t s);
// The flat tile list of positions [T0, T1) from the CSR (row_ptr, entries): per (g, b)
// the list's positions cut into tiles of 16 ppr positions, tile_off[G*nb] = total
// tiles; tile i is records [i ppr, (i + 1) ppr) of rec.
cudaError_t launch_tile_schedule(const int32_t* row_ptr, const int32_t* entries, int64_t N, int G, int k, int64_t nb,
                                 int64_t T0, int64_t T1, int64_t max_tiles, int ppr, int32_t* lo, int32_t* cnt,
                                 int32_t* tiles, int32_t* tile_off, TileRecord* rec, cudaStream_t s);
cudaError_t launch_attn(const void* q, const void* k, const void* v, const int32_t* block_idx, const AttnPlan& p,
                        float scale, void* out, float* lse, void* scratch, DeviceStatus* st, cudaStream_t s);
// The select kernel followed by the attention call, on one stream.
cudaError_t launch_prefill(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                           int d_I, const AttnPlan& p, float scale, int32_t* block_idx, void* out, float* lse,
                           void* scratch, DeviceStatus* st, cudaStream_t s, bool f8 = false,
                           const int32_t* blk_lo = nullptr);

// ---- backward (msa_bwd.cu)
size_t bwd_scratch_bytes(int64_t N, int H_q, int H_kv, int d, int Bk, int k);
// Gradients are fp32 and accumulated in place (the launcher clears them first).
cudaError_t launch_bwd(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                       const int32_t* block_idx, const void* out, const float* lse, const void* dout, int64_t N,
                       int H_q, int H_kv, int d, int d_I, int Bk, int kb, float scale, float kl_weight, float* dq,
                       float* dk, float* dv, float* dq_idx, float* dk_idx, float* kl, void* scratch, DeviceStatus* st,
                       cudaStream_t s);

// ---- warmup mode (msa_warmup.cu)
// fwd: out, lse (dense causal attention) and lseI [G, N] (the index branch's
// lse over every key j <= t); grad: kl [G, N], dq_idx [N, G, d_I] and dk_idx
// [N, d_I] (cleared here, then accumulated) from lse and lseI.
cudaError_t launch_warmup(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx, int64_t N,
                          int H_q, int H_kv, int d, int d_I, float scale, float kl_weight, bool fwd, bool grad,
                          void* out, float* lse, float* lseI, float* dq_idx, float* dk_idx, float* kl, cudaStream_t s);

// ---- warmup mode on tcgen05 (msa_warmup_tc.cu): d = d_I = 128 and gs = 8
bool warmup_tc_supported(int d, int d_I, int H_q, int H_kv);
// out, lse (dense causal attention) and lseI; st may be null.
cudaError_t launch_warmup_fwd_tc(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                                 int64_t N, int H_q, int H_kv, float scale, void* out, float* lse, float* lseI,
                                 DeviceStatus* st, cudaStream_t s);
// kl, dq_idx and dk_idx are cleared here, then accumulated; st may be null.
cudaError_t launch_warmup_grad_tc(const void* q, const void* k, const void* q_idx, const void* k_idx, int64_t N,
                                  int H_q, int H_kv, float scale, float kl_weight, const float* lse, const float* lseI,
                                  float* dq_idx, float* dk_idx, float* kl, DeviceStatus* st, cudaStream_t s);

// ---- decode (msa_decode.cu)
// Where token `key` of sequence `seq` sits in a decode cache: contiguous (no
// table: row seq * ctx_max + key) or paged (row table[seq][key / page] * page +
// key % page of a pool of n_pages pages; page a multiple of 16 tokens).
struct CacheMap {
  const int32_t* table = nullptr;  // [B, max_pages] physical page of each logical page
  int64_t max_pages = 0;
  int64_t n_pages = 0;
  int page = 0;
#ifdef __CUDACC__
  // a page id outside [0, n_pages) sets the device error word and reads page 0
  __device__ __forceinline__ int64_t row(int64_t seq, int64_t key, DeviceStatus* st) const;
#endif
};
struct DecodePlan {
  int B;
  int64_t ctx_max;
  int H_q, H_kv, d, d_I, Bk, k, gs;
  int splits;          // CTAs per sequence in the index-key scan
  int max_cta_blocks;  // candidate blocks of one scan CTA, at most
  bool f8 = false;     // index query and index-key cache hold FP8 E4M3 codes
};
DecodePlan decode_plan(int B, int64_t ctx_max, int H_q, int H_kv, int d, int d_I, int Bk, int k);
size_t decode_scratch_bytes(const DecodePlan& p);
// Bytes at the start of the decode scratch that must be zero when a call starts
// (the completion tickets of the attention CTAs).
size_t decode_clear_bytes(const DecodePlan& p);
cudaError_t launch_decode(const void* q_t, const void* q_idx_t, const void* k_idx_cache, const void* k_cache,
                          const void* v_cache, const int32_t* ctx_len, const DecodePlan& p, float scale, void* out,
                          float* lse, int32_t* block_idx, void* scratch, DeviceStatus* st, cudaStream_t s,
                          const CacheMap* paged = nullptr);

// Fixed device scratch of msa_decode_noalloc (8 MiB, shared by all calls on a
// device).  Returns its device address for the current device (looked up on
// the first call per device), or an error if `need` exceeds it.
constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;
cudaError_t noalloc_scratch(size_t need, void** out);

}  // namespace msa
