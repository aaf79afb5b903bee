/*
 * msa.h — C ABI of libmsa.so, the GB300 (sm_103a) forward path of MiniMax
 * Sparse Attention (MSA).
 *
 * The method (pages: the "MSA" study note, sections 2-1 "Two-branch sparse
 * attention" and 2-3 "Fixed attention budget"; the chipsbuilder.com article,
 * "Funzionamento Delle Due Branch"):
 *   index scores  s[t,g,j] = q^I[t,g] . k^I[j] / sqrt(d_I)      (j <= t)
 *   block scores  S[t,g,b] = max over j in block b, j <= t, of s[t,g,j]
 *   block set     B[t,g]   = {local(t)} + the k-1 best S[t,g,b], b < local(t)
 *   output        O[t,h]   = softmax(scale * q[t,h] K_J^T) V_J,
 *                 J = tokens j <= t of the blocks in B[t, g(h)], g(h) = h / (H_q/H_kv)
 *
 * Conventions for every call:
 *   - Returns a status; work is enqueued asynchronously on `stream`.
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; the
 *     library neither frees nor keeps it after the call returns.
 *   - The library allocates nothing.  Scratch comes from a caller-owned device
 *     workspace whose minimum size the matching *_workspace() call returns.
 *     The workspace must stay alive and untouched until the enqueued work has
 *     finished; two calls in flight at once need two workspaces.
 *   - Tensors are dense, row-major, contiguous; bf16 is stored as 16-bit
 *     words; shapes are given beside each argument.
 *   - Indices are 0-based.  local(t) = t / Bk.  nb = ceil(N / Bk).
 *   - Host-side validation happens before any launch and returns
 *     MSA_ERR_INVALID_ARGUMENT (bad pointer, size or shape),
 *     MSA_ERR_UNSUPPORTED (a valid shape outside the supported set) or
 *     MSA_ERR_WORKSPACE_TOO_SMALL.  A failed launch returns MSA_ERR_CUDA.
 *   - Bad data found on the device (a block id outside [0, nb) other than -1)
 *     does not trap: the entry is skipped and an error word at the start of
 *     the workspace is set.  msa_check_device_error() reads that word; each
 *     call clears it when it starts.
 *
 * Supported shapes: d in {64, 128}; d_I in {32, 64, 128}; Bk in {64, 128};
 * 1 <= k <= 32; H_q / H_kv in {1, 2, 4, 8}; 1 <= H_kv <= 64; N >= 1.
 */
#ifndef MSA_H
#define MSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* msa_stream_t; /* same type as cudaStream_t; NULL = legacy default stream */

typedef enum {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARGUMENT = 1,
  MSA_ERR_UNSUPPORTED = 2,
  MSA_ERR_WORKSPACE_TOO_SMALL = 3,
  MSA_ERR_CUDA = 4,
  MSA_ERR_BAD_INDEX = 5,
  MSA_ERR_TIMEOUT = 6
} msa_status_t;

/* Problem shape.  G = H_kv GQA groups (one index-query head per group);
 * gs = H_q / H_kv query heads per group; k counts the local block. */
typedef struct {
  int64_t N; /* tokens (prefill) or cache capacity per sequence (decode) */
  int H_q;   /* query heads */
  int H_kv;  /* key/value heads = GQA groups = index-query heads */
  int d;     /* head dim of q, k, v */
  int d_I;   /* index head dim of q^I, k^I */
  int Bk;    /* tokens per KV block */
  int k;     /* blocks per (query, group), local block included */
} msa_shape_t;

/* ---------------------------------------------------------------- select
 * Index branch: scoring, block max-pooling and the local-pinned top-k.
 * Pages: "MSA" study note 2-3 (equations for s, S and the block set), 3-2
 * "Index Branch", 3-4 "Forced local block", 3-5 "GPU kernel co-design"
 * (exp-free top-k on raw scores); Flash-MSA "プロキシアテンション" (streaming
 * top-k while sweeping key tiles; local block pinned to +inf).
 *
 *   q_idx     [N, G, d_I] bf16: index queries (one head per group)
 *   k_idx     [N, d_I]    bf16: index keys (one head shared by all groups)
 *   block_idx [G, N, k]   int32 out: slot 0 = local(t); slots 1.. = the
 *             min(k-1, local(t)) blocks b < local(t) of largest S, in
 *             descending S, equal S ordered by ascending b (the lower block
 *             wins a tie at the cut); remaining slots = -1.
 * Ranking uses the fp32 tensor-core dot products q^I . k^I (a positive
 * scale does not change the order).
 */
size_t msa_select_blocks_workspace(int64_t N, int G, int d_I, int Bk, int k);
msa_status_t msa_select_blocks(const void* q_idx, const void* k_idx, int64_t N, int G, int d_I, int Bk,
                               int k, int32_t* block_idx, void* workspace, size_t workspace_bytes,
                               msa_stream_t stream);

/* ---------------------------------------------------------------- invert
 * B -> B*: for every group g and block b, the (t, slot) pairs whose set
 * holds b.  Pages: Flash-MSA "バックワードパス" (B[batch, head, query,
 * slot] -> block inverted to B*[batch, head, block] -> queries) and the
 * "MSA" study note 3-5 (reverse sparse index feeding KV-outer attention).
 *
 *   block_idx [G, N, k] int32 (ids in [0, nb) or -1)
 *   row_ptr   [G, nb+1] int32 out: offsets into the group's entry region
 *   entries   [G, N*k]  int32 out: group g's list of block b is
 *             entries[g*N*k + row_ptr[g][b] .. g*N*k + row_ptr[g][b+1]),
 *             each entry t*k + slot, in ascending t (deterministic).
 *             Entries past n_entries[g] are left untouched.
 *   n_entries [G]       int32 out: entries listed for group g.
 * An id outside [0, nb) other than -1 sets the device error word and is not
 * listed.
 */
size_t msa_invert_blocks_workspace(int64_t N, int G, int Bk, int k);
msa_status_t msa_invert_blocks(const int32_t* block_idx, int64_t N, int G, int Bk, int k, int32_t* row_ptr,
                               int32_t* entries, int32_t* n_entries, void* workspace, size_t workspace_bytes,
                               msa_stream_t stream);

/* ---------------------------------------------------------------- attend
 * Main branch: exact softmax attention over the selected blocks' causally
 * visible tokens, every head of group g reading group g's set, computed
 * KV-outer (each K/V block once per tile of the queries that chose it) with
 * per-(t, h, slot) partial results merged by their log-sum-exp.
 * Pages: "MSA" study note 2-3 (Attn over K_{g,B}, V_{g,B}), 3-3 "Main
 * Branch", 3-5 (KV-outer execution, pre-scheduled tile chunking, two-phase
 * combine, LSE kept); chipsbuilder "Funzionamento Delle Due Branch" (tokens
 * causally visible in the selected blocks); Flash-MSA "フォワードパス" (main
 * LSE saved).
 *
 *   q         [N, H_q, d]  bf16
 *   k, v      [N, H_kv, d] bf16
 *   block_idx [G, N, k]    int32: each row's set (-1 = empty slot; a repeated
 *             id counts once; ids past local(t) hold no visible token and add
 *             nothing)
 *   scale     softmax scale (1/sqrt(d) in the pages)
 *   out       [N, H_q, d]  bf16 out: O[t, h]
 *   lse       [H_q, N]     fp32 out: natural-log log-sum-exp of the scaled
 *             scores over J; -inf (with out = 0) when J is empty.
 */
size_t msa_sparse_attn_fwd_workspace(const msa_shape_t* shape);
msa_status_t msa_sparse_attn_fwd(const void* q, const void* k, const void* v, const int32_t* block_idx,
                                 const msa_shape_t* shape, float scale, void* out, float* lse,
                                 void* workspace, size_t workspace_bytes, msa_stream_t stream);

/* ---------------------------------------------------------------- backward
 * Gradients of msa_sparse_attn_fwd (main branch) and of the index branch's KL
 * alignment loss, over the same block sets.  Pages: "MSA" study note 4-2 (the
 * index branch learns from a KL loss against the mean of the GQA group's
 * main-branch attention probabilities) and 4-3 (the teacher is detached and the
 * index input gets a stop-gradient: the KL reaches only q^I and k^I);
 * Flash-MSA "バックワードパス" (both backward passes over the cached sparse
 * blocks, scheduled through the inverted map B*) and "KLダイバージェンス損失"
 * (the gradient on the index logits is index probability minus teacher).
 *
 * Per row (t, h), group g = h / gs, J = the selected blocks' tokens j <= t:
 *   P_j = exp(scale q.k_j - lse), D = dout.out, dZ_j = P_j (dout.v_j - D),
 *   dq = scale sum_j dZ_j k_j, dk_j += scale dZ_j q, dv_j += P_j dout.
 * Per row (t, g): teacher pbar_j = mean over the group's heads of P_j; index
 * logits z_j = q^I.k^I_j / sqrt(d_I); p_j = softmax over J of z;
 *   kl[g, t] = sum_j pbar_j (log pbar_j - log p_j)
 *   (loss = kl_weight * sum over (t, g) of kl), dL/dz_j = kl_weight (p_j - pbar_j),
 *   dq_idx = sum_j dL/dz_j k^I_j / sqrt(d_I), dk_idx_j += dL/dz_j q^I / sqrt(d_I).
 *
 *   q, k, v, q_idx, k_idx, block_idx, scale: as the forward calls
 *   out, lse  the forward's outputs for the same inputs
 *   dout      [N, H_q, d] bf16: gradient of the loss with respect to out
 *   dq        [N, H_q, d] fp32 out;  dk, dv [N, H_kv, d] fp32 out
 *   dq_idx    [N, G, d_I] fp32 out;  dk_idx [N, d_I] fp32 out
 *   kl        [G, N] fp32 out (nullable): each row's KL
 *   workspace msa_sparse_attn_bwd_workspace(shape) bytes, 256-byte aligned;
 *             it grows with N * G * k (the B* entries and per-slot partials)
 *             plus a teacher buffer bounded by query slabs of at most 131072
 *             positions (G * k * Bk * 2 bytes a position of one slab)
 * The gradient outputs are cleared and then accumulated in place on `stream`.
 */
size_t msa_sparse_attn_bwd_workspace(const msa_shape_t* shape);
msa_status_t msa_sparse_attn_bwd(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                                 const int32_t* block_idx, const void* out, const float* lse, const void* dout,
                                 const msa_shape_t* shape, float scale, float kl_weight, float* dq, float* dk,
                                 float* dv, float* dq_idx, float* dk_idx, float* kl, void* workspace,
                                 size_t workspace_bytes, msa_stream_t stream);

/* ---------------------------------------------------------------- warmup mode
 * The training-time variant that comes before sparse routing.  Pages: the
 * "MSA" study note, 4-4 "Indexer warmup" (the main branch runs full attention
 * while the index branch learns the KL alignment against the full-context
 * teacher; top-k routing is switched on afterwards), 4-2 and 4-3 (the teacher
 * is the mean of the group's main-branch probabilities, detached, and the KL
 * reaches only q^I and k^I), 1-1 (dense causal GQA attention).  Same
 * definitions as msa_sparse_attn_bwd's index branch, with J(t, g) = every key
 * j <= t.  shape->Bk and shape->k must be valid values but are not used.  No
 * workspace and no device-side error paths.
 *
 * msa_warmup_fwd: dense causal attention and the index branch's normaliser.
 *   q, k, v, q_idx, k_idx: as msa_prefill
 *   out      [N, H_q, d] bf16 out: softmax(scale q.k_j, j <= t) V
 *   lse      [H_q, N] fp32 out: natural-log log-sum-exp of the scaled scores
 *   lse_idx  [G, N] fp32 out: log-sum-exp over j <= t of q^I.k^I_j / sqrt(d_I)
 * msa_warmup_index_grad: the KL loss of every row and its gradients, from the
 *   forward's lse and lse_idx.
 *   kl       [G, N] fp32 out: KL(teacher || index) of each row (not weighted)
 *   dq_idx   [N, G, d_I] fp32 out: kl_weight * d(sum KL)/d q^I
 *   dk_idx   [N, d_I] fp32 out: kl_weight * d(sum KL)/d k^I (overwritten)
 */
msa_status_t msa_warmup_fwd(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                            const msa_shape_t* shape, float scale, void* out, float* lse, float* lse_idx,
                            msa_stream_t stream);
msa_status_t msa_warmup_index_grad(const void* q, const void* k, const void* q_idx, const void* k_idx,
                                   const float* lse, const float* lse_idx, const msa_shape_t* shape, float scale,
                                   float kl_weight, float* dq_idx, float* dk_idx, float* kl, msa_stream_t stream);

/* ---------------------------------------------------------------- prefill
 * The whole forward pass in one call: msa_select_blocks followed by
 * msa_sparse_attn_fwd on the same shapes and stream, with the same results.
 * Pages: "MSA" study note 3-5 (the index and main branches as separate
 * kernels feeding KV-outer attention and the two-phase combine); the pages
 * give no fused entry point.
 *
 *   q, k, v, q_idx, k_idx, scale, out, lse: as msa_select_blocks and
 *             msa_sparse_attn_fwd
 *   block_idx [G, N, k] int32 out: the sets, as msa_select_blocks
 *   workspace msa_prefill_workspace(shape) bytes, 256-byte aligned (one
 *             workspace serves both stages)
 */
size_t msa_prefill_workspace(const msa_shape_t* shape);
msa_status_t msa_prefill(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                         const msa_shape_t* shape, float scale, int32_t* block_idx, void* out, float* lse,
                         void* workspace, size_t workspace_bytes, msa_stream_t stream);

/* ---------------------------------------------------------------- varlen prefill
 * Several sequences in one prefill, each in its own run of cells.  Pages:
 * velog llama.cpp analysis, section 4 (with sequences mixed in one shared
 * cache the condition "block of the sequence = run of consecutive cache
 * cells" breaks and the port falls back to dense attention) and section 5
 * (the fix named there: an explicit per-sequence position -> cell -> block
 * map).
 *
 * Layout: sequence s holds cells [cu_seqlens[s], cu_seqlens[s+1]) of the
 * N-cell tensors (q, k, v, q_idx, k_idx, out, lse, block_idx: the msa_prefill
 * layouts with N cells); its position p is cell cu_seqlens[s] + p.  Every
 * cu_seqlens[s] is a multiple of Bk, cu_seqlens[0] = 0, the values do not
 * decrease and cu_seqlens[S] <= N.  A sequence's blocks are therefore whole
 * runs of cells and never shared.  Cells of a sequence past its last token
 * (padding up to the next block boundary) and cells past cu_seqlens[S] are
 * computed like tokens; no real token selects or attends to them (they lie
 * after every token of their block, and blocks of other sequences are never
 * candidates).
 *
 * Per cell t of sequence s the set is msa_select_blocks' rule with the
 * candidates restricted to the sequence: {local(t)} plus the k-1 best blocks b
 * with cu_seqlens[s]/Bk <= b < local(t).  Block ids are cell block ids.  The
 * attention is msa_sparse_attn_fwd on those sets, so out and lse of every
 * real token equal msa_prefill run on that sequence alone (block ids offset
 * by cu_seqlens[s]/Bk).
 *
 *   cu_seqlens [S+1] int32 (device), S >= 1.  A cu_seqlens that breaks the
 *              rules above sets the device error word (MSA_ERR_BAD_INDEX from
 *              msa_check_device_error); every cell then keeps only its local
 *              block.
 *   workspace  msa_select_blocks_varlen_workspace() / msa_prefill_varlen_workspace() bytes
 */
size_t msa_select_blocks_varlen_workspace(int64_t N, int G, int d_I, int Bk, int k);
msa_status_t msa_select_blocks_varlen(const void* q_idx, const void* k_idx, const int32_t* cu_seqlens, int S,
                                      int64_t N, int G, int d_I, int Bk, int k, int32_t* block_idx, void* workspace,
                                      size_t workspace_bytes, msa_stream_t stream);
size_t msa_prefill_varlen_workspace(const msa_shape_t* shape);
msa_status_t msa_prefill_varlen(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                                const int32_t* cu_seqlens, int S, const msa_shape_t* shape, float scale,
                                int32_t* block_idx, void* out, float* lse, void* workspace, size_t workspace_bytes,
                                msa_stream_t stream);

/* ---------------------------------------------------------------- decode
 * One decode step for B sequences.  The query of sequence s sits at position
 * t = ctx_len[s] - 1 and its k, v and k^I are already in the caches.  The
 * whole index-key cache is scanned (the only part that grows with the
 * context), the block set is chosen as in msa_select_blocks, and only the
 * selected K/V blocks are read.  Pages: velog llama.cpp analysis, section 2
 * (256 B/token index-key scan, fixed K/V read per step) and section 4 (block
 * scores, max-pooling, forced local block, top-k, then attention over the
 * gathered blocks).
 *
 *   q_t          [B, H_q, d] bf16
 *   q_idx_t      [B, G, d_I] bf16
 *   k_idx_cache  [B, shape->N, d_I] bf16  (shape->N = cache capacity)
 *   k_cache      [B, shape->N, H_kv, d] bf16, v_cache likewise
 *   ctx_len      [B] int32 (device): 1 <= ctx_len[s] <= shape->N
 *   out          [B, H_q, d] bf16 out
 *   lse          [B, H_q] fp32 out (nullable)
 *   block_idx    [B, G, k] int32 out (nullable): the sets chosen
 * ctx_len values outside [1, N] set the device error word; that sequence's
 * outputs are zero.
 */
size_t msa_decode_workspace(int B, const msa_shape_t* shape);
msa_status_t msa_decode(const void* q_t, const void* q_idx_t, const void* k_idx_cache, const void* k_cache,
                        const void* v_cache, const int32_t* ctx_len, int B, const msa_shape_t* shape, float scale,
                        void* out, float* lse, int32_t* block_idx, void* workspace, size_t workspace_bytes,
                        msa_stream_t stream);

/* ---------------------------------------------------------------- paged decode
 * msa_decode over caches kept in pages: sequence s's token j is row
 * page_table[s][j / page_size] * page_size + j % page_size of the page pools,
 * so sequences of different lengths share one pool without a dense
 * [B, capacity] layout.  Same selection, attention and outputs as msa_decode
 * on the caches the pages spell out.  Pages: velog llama.cpp analysis, section
 * 4 (a per-sequence position -> cache cell -> block map is what lets a decode
 * kernel serve several sequences of different lengths, where the analysed
 * port falls back to one dense unified cache).
 *
 *   k_idx_pool  [n_pages, page_size, d_I] bf16
 *   k_pool      [n_pages, page_size, H_kv, d] bf16, v_pool likewise
 *   page_table  [B, max_pages] int32 (device): physical page of each logical
 *               page; entries past a sequence's ctx_len are not read
 *   page_size   tokens per page, a positive multiple of 16
 *   shape->N    = max_pages * page_size (a sequence's capacity)
 *   workspace   msa_decode_workspace(B, shape) bytes
 *   the rest as msa_decode.
 * A page id read outside [0, n_pages) sets the device error word (reported as
 * MSA_ERR_BAD_INDEX) and page 0 is read in its place.
 */
msa_status_t msa_decode_paged(const void* q_t, const void* q_idx_t, const void* k_idx_pool, const void* k_pool,
                              const void* v_pool, const int32_t* page_table, int64_t max_pages, int64_t n_pages,
                              int page_size, const int32_t* ctx_len, int B, const msa_shape_t* shape, float scale,
                              void* out, float* lse, int32_t* block_idx, void* workspace, size_t workspace_bytes,
                              msa_stream_t stream);

/* ---------------------------------------------------------------- FP8 index inputs
 * The index branch on FP8 inputs.  Pages: the chipsbuilder.com article, "Co-
 * Design Del Kernel" (FP8 is among the precisions of the method's kernel),
 * and the "MSA" study note, 6 "Limitations" item 1 (the index branch scores
 * the whole context, so its inputs carry the cost that grows with it).
 *
 * FP8 here is E4M3 of the OCP 8-bit floating point specification: one byte
 * per element, 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no
 * infinity, largest finite magnitude 448.  The selection rule is exactly that
 * of msa_select_blocks, applied to the decoded values: every product of two
 * E4M3 values is exact and the tensor cores sum them in fp32.  Multiplying all
 * of q^I, or all of k^I, by one positive factor before quantizing changes no
 * ranking, so the selection calls take no scale.  Supported d_I: 64 or 128
 * (MSA_ERR_UNSUPPORTED otherwise).
 *
 * msa_quantize_e4m3: y[i] = the E4M3 code nearest to the fp32 product
 *   (bf16 x[i]) * scale, ties to the even code, magnitudes beyond 448
 *   saturated to 448, NaN kept NaN.  x [n] bf16 (2-byte aligned), y [n] bytes
 *   out; no workspace.
 * msa_select_blocks_fp8: msa_select_blocks with q_idx [N, G, d_I] and
 *   k_idx [N, d_I] as E4M3 codes; workspace msa_select_blocks_workspace().
 * msa_prefill_fp8: msa_prefill with E4M3 q_idx and k_idx (q, k, v stay bf16);
 *   workspace msa_prefill_workspace().
 * msa_decode_fp8: msa_decode with q_idx_t [B, G, d_I] and k_idx_cache
 *   [B, N, d_I] as E4M3 codes, so the scan reads d_I bytes per cached token
 *   instead of 2 d_I; workspace msa_decode_workspace().
 * msa_decode_paged_fp8: msa_decode_paged with E4M3 q_idx_t and k_idx_pool
 *   [n_pages, page_size, d_I].
 */
msa_status_t msa_quantize_e4m3(const void* x, int64_t n, float scale, void* y, msa_stream_t stream);
msa_status_t msa_select_blocks_fp8(const void* q_idx, const void* k_idx, int64_t N, int G, int d_I, int Bk, int k,
                                   int32_t* block_idx, void* workspace, size_t workspace_bytes, msa_stream_t stream);
msa_status_t msa_prefill_fp8(const void* q, const void* k, const void* v, const void* q_idx, const void* k_idx,
                             const msa_shape_t* shape, float scale, int32_t* block_idx, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, msa_stream_t stream);
msa_status_t msa_decode_fp8(const void* q_t, const void* q_idx_t, const void* k_idx_cache, const void* k_cache,
                            const void* v_cache, const int32_t* ctx_len, int B, const msa_shape_t* shape, float scale,
                            void* out, float* lse, int32_t* block_idx, void* workspace, size_t workspace_bytes,
                            msa_stream_t stream);
msa_status_t msa_decode_paged_fp8(const void* q_t, const void* q_idx_t, const void* k_idx_pool, const void* k_pool,
                                  const void* v_pool, const int32_t* page_table, int64_t max_pages, int64_t n_pages,
                                  int page_size, const int32_t* ctx_len, int B, const msa_shape_t* shape, float scale,
                                  void* out, float* lse, int32_t* block_idx, void* workspace, size_t workspace_bytes,
                                  msa_stream_t stream);

/* ---------------------------------------------------------------- decode without allocation
 * The same decode step as msa_decode, for callers that cannot allocate device
 * memory: for instance a plugin whose host application owns every byte of the
 * GPU, or a serving loop that must not call cudaMalloc because it can block
 * and synchronize the device mid-step.  The pages have no counterpart of this
 * call; it exists only for such callers.
 *
 * No workspace argument: the scratch is a fixed 8 MiB array that the library
 * keeps in device memory on every GPU that loads it, until the process exits.
 * The call makes no allocation of any kind (no cudaMalloc/cudaFree, no
 * allocating library routine).  Arguments, layouts and outputs are those of
 * msa_decode.
 *   - The first call on a device looks up the array's device address for that
 *     device (cudaGetSymbolAddress, with the device current); make that first
 *     call before any stream capture.  The address is kept per device and
 *     context: a call made after cudaDeviceReset, or under another context of
 *     the same device, looks it up again, so it is never stale.
 *   - Shapes whose scratch (what msa_decode_workspace() reports for them)
 *     exceeds 8 MiB are rejected with MSA_ERR_WORKSPACE_TOO_SMALL before any
 *     launch.  B = 4, H_q = 64, H_kv = 8, d = 128, k = 16 needs about 2.4 MiB.
 *   - All calls on a device share the one array and it keeps the previous
 *     call's contents; each call clears what must start at zero.  Two calls
 *     that can overlap on the GPU (different streams, or different host
 *     threads) race on it: order them on one stream.
 *   - Device-side bad data (ctx_len outside [1, N]) still zeroes that
 *     sequence's outputs, and a bounded device wait that gives up still ends
 *     its kernel cleanly, but both flags live in the shared array's status
 *     word: this call returns MSA_OK for them and cannot report
 *     MSA_ERR_BAD_INDEX or MSA_ERR_TIMEOUT.  Callers that need those statuses
 *     use msa_decode with a workspace and msa_check_device_error.
 */
msa_status_t msa_decode_noalloc(const void* q_t, const void* q_idx_t, const void* k_idx_cache, const void* k_cache,
                                const void* v_cache, const int32_t* ctx_len, int B, const msa_shape_t* shape,
                                float scale, void* out, float* lse, int32_t* block_idx, msa_stream_t stream);

/* ---------------------------------------------------------------- status
 * msa_check_device_error: waits for `stream`, then returns MSA_ERR_BAD_INDEX
 * if the last call that used `workspace` met bad data on the device,
 * MSA_ERR_TIMEOUT if one of its kernels gave up a bounded wait, MSA_OK
 * otherwise (or MSA_ERR_CUDA if the wait itself failed).
 * msa_status_string: a static, readable description of a status.
 */
msa_status_t msa_check_device_error(void* workspace, msa_stream_t stream);
const char* msa_status_string(msa_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H */
