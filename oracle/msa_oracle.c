/*
 * ORACLE — test infrastructure only.  Plain, slow fp64 CPU statement of the
 * MiniMax Sparse Attention (MSA) forward path and of its backward.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load this library; the
 * product path never does.  It shares no code with the CUDA library.
 *
 * Sources (page titles and sections):
 *   [P1] "MSA" study note (dimensionstp.github.io), 1-1 "Full attention의 병목"
 *        (dense causal GQA softmax, scale 1/sqrt(d_h)); 2-1 "Two-branch sparse
 *        attention" (the four steps); 2-3 "Fixed attention budget" (equations
 *        for s, S and the selected set; Bk = 128, k = 16 including the local
 *        block -> at most 2048 keys); 3-2 "Index Branch" (max-pooling of the
 *        causally visible token scores); 3-3 "Main Branch" (exact softmax over
 *        the selected support, per-head weights, group-shared selection); 3-4
 *        "Forced local block"; 3-5 "GPU kernel co-design" (exp-free top-k;
 *        LSE saved).
 *   [P2] "MSA: un nuovo approccio all'attenzione sparsa" (chipsbuilder.com),
 *        "Che cos'é MSA" (k = 16 blocks incl. the query's block, kBk = 2048)
 *        and "Funzionamento Delle Due Branch" (one index query head per GQA
 *        group, one shared index key head; causally visible tokens).
 *   [P3] "MiniMax M3의 Sparse Attention 구조 및 llama.cpp 구현 제약 분석"
 *        (velog.io), section 2 (decode: the whole index-key cache is scanned,
 *        only the selected K/V blocks are read).
 *   [P4] "Flash-MSA" (hackernews.jp translation), "フォワードパス" / "プロキシ
 *        アテンション" (top-k on raw scores while streaming keys; the local
 *        block's score set to +inf; main LSE saved) and "バックワードパス"
 *        (the block->query inversion B -> B*).
 *
 * Readings where the pages leave a step open:
 *   - k counts the local block: the set is {local(t)} plus the (k-1)
 *     highest-scoring blocks b < local(t) ([P1] 2-3, [P2], [P4] +inf pin);
 *   - fewer than k-1 earlier blocks: all of them are taken (set size
 *     min(k, local(t)+1)); unused slots hold -1;
 *   - equal block scores: the lower block index wins;
 *   - slot 0 = local(t), then descending score (ties by ascending block);
 *   - lse is the natural-log log-sum-exp of the scaled main scores;
 *   - decode: the query sits at position ctx_len-1 and its keys are already
 *     in the caches.
 *
 * Backward (msa_ref_sparse_attn_bwd, at the end of this file):
 *   [P1] 4-2 "Why LM loss alone is insufficient" (the index branch learns from
 *        an auxiliary KL loss whose teacher is the mean over the GQA group's
 *        query heads of the main-branch attention probabilities), 4-3
 *        "Gradient detach" (the teacher is detached and the index input gets a
 *        stop-gradient: the KL updates only the index query and key);
 *   [P4] "バックワードパス" (main and proxy gradients over the cached sparse
 *        blocks; proxy LSE recomputed over the selected blocks) and "KL
 *        ダイバージェンス損失" (the KL gradient on the proxy logits is the proxy
 *        probability minus the main probability).
 *   Readings: the KL of row (t, g) is taken over the same support J(t, g) as
 *   the main attention (the selected blocks' visible tokens) with the index
 *   logits q^I.k^I / sqrt(d_I); the loss is kl_weight * sum over (t, g) of
 *   KL(teacher || index); the main branch receives dO only.
 *
 * Arithmetic: bf16 (or FP8 E4M3) inputs widened exactly to double; every
 * dot product, maximum, exponential and sum in double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEM 2

/* ------------------------------------------------------------------ helpers */
static double bf16_to_double(uint16_t h) {
  union { uint32_t u; float f; } c;
  c.u = (uint32_t)h << 16;
  return (double)c.f;
}

static double dot_bf16(const uint16_t* a, const uint16_t* b, int n) {
  double s = 0.0;
  for (int i = 0; i < n; ++i) s += bf16_to_double(a[i]) * bf16_to_double(b[i]);
  return s;
}

typedef struct {
  int64_t lo, hi;
  void* ctx;
  void (*fn)(int64_t, void*);
} range_t;

static void* range_main(void* p) {
  range_t* r = (range_t*)p;
  for (int64_t i = r->lo; i < r->hi; ++i) r->fn(i, r->ctx);
  return NULL;
}

/* Runs fn(i) for i in [0, n) over n_threads threads (interleaved chunks). */
static void parallel_for(int64_t n, int n_threads, void (*fn)(int64_t, void*), void* ctx) {
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 512) n_threads = 512;
  if ((int64_t)n_threads > n) n_threads = (int)(n > 0 ? n : 1);
  pthread_t th[512];
  range_t rg[512];
  for (int i = 0; i < n_threads; ++i) {
    rg[i].lo = n * i / n_threads;
    rg[i].hi = n * (i + 1) / n_threads;
    rg[i].ctx = ctx;
    rg[i].fn = fn;
  }
  for (int i = 1; i < n_threads; ++i) pthread_create(&th[i], NULL, range_main, &rg[i]);
  range_main(&rg[0]);
  for (int i = 1; i < n_threads; ++i) pthread_join(th[i], NULL);
}

/* ------------------------------------------------- step 1: block scores S */
/*
 * [P1] 2-3: s_{t,g,j} = q^I_{t,g} . k^I_j / sqrt(d_I) and
 * S_{t,g,b} = max over j in block b with j <= t of s_{t,g,j}.
 * Blocks past local(t) have no visible token: S = -inf there.
 */
static void block_scores_row(const uint16_t* qrow /*[d_I]*/, const uint16_t* k_idx, int64_t t,
                             int d_I, int Bk, int64_t nb, double* S /*[nb]*/) {
  double inv = 1.0 / sqrt((double)d_I);
  double q[512];
  for (int c = 0; c < d_I; ++c) q[c] = bf16_to_double(qrow[c]);
  for (int64_t b = 0; b < nb; ++b) S[b] = -INFINITY;
  /* four keys at a time: four independent dot products, each summed in order */
  int64_t j = 0;
  for (; j + 3 <= t; j += 4) {
    const uint16_t *k0 = k_idx + j * d_I, *k1 = k0 + d_I, *k2 = k1 + d_I, *k3 = k2 + d_I;
    double s0 = 0.0, s1 = 0.0, s2 = 0.0, s3 = 0.0;
    for (int c = 0; c < d_I; ++c) {
      s0 += q[c] * bf16_to_double(k0[c]);
      s1 += q[c] * bf16_to_double(k1[c]);
      s2 += q[c] * bf16_to_double(k2[c]);
      s3 += q[c] * bf16_to_double(k3[c]);
    }
    double s[4] = {s0 * inv, s1 * inv, s2 * inv, s3 * inv};
    for (int i = 0; i < 4; ++i) {
      int64_t b = (j + i) / Bk;
      if (s[i] > S[b]) S[b] = s[i];
    }
  }
  for (; j <= t; ++j) {
    double s = dot_bf16(qrow, k_idx + j * d_I, d_I) * inv;
    int64_t b = j / Bk;
    if (s > S[b]) S[b] = s;
  }
}

/*
 * Step 2 ([P1] 2-3, 3-4, 3-5; [P4] +inf pin): slot 0 = local(t); then the
 * k-1 largest S over b < local(t), ties to the lower b, in descending order;
 * then -1.  kth[0], kth[1] = the (k-1)-th and k-th largest non-local scores
 * (the last taken and the first left out), +inf/-inf when no block is left
 * out.
 */
static void topk_row(const double* S, int64_t t, int Bk, int k, int32_t* out /*[k]*/,
                     double* kth /*[2] or NULL*/, unsigned char* taken /*[nb] scratch*/) {
  int64_t local = t / Bk;
  for (int i = 0; i < k; ++i) out[i] = -1;
  out[0] = (int32_t)local;
  for (int64_t b = 0; b < local; ++b) taken[b] = 0;
  double last = INFINITY;
  int n_take = (int)((local < (int64_t)(k - 1)) ? local : (int64_t)(k - 1));
  for (int i = 0; i < n_take; ++i) {
    int64_t best = -1;
    for (int64_t b = 0; b < local; ++b) {
      if (taken[b]) continue;
      if (best < 0 || S[b] > S[best]) best = b; /* strict: the lower b keeps a tie */
    }
    taken[best] = 1;
    out[1 + i] = (int32_t)best;
    last = S[best];
  }
  if (kth) {
    double next = -INFINITY;
    for (int64_t b = 0; b < local; ++b)
      if (!taken[b] && S[b] > next) next = S[b];
    kth[0] = (n_take > 0) ? last : INFINITY;
    kth[1] = next;
  }
}

typedef struct {
  const uint16_t* q_idx_rows; /* [n_rows, G, d_I] */
  const uint16_t* k_idx;      /* [N, d_I] */
  const int64_t* rows;
  int64_t n_rows, N, nb;
  int G, d_I, Bk, k;
  double* S;        /* [n_rows, G, nb] or NULL */
  int32_t* blk;     /* [G, n_rows, k] or NULL */
  double* kth;      /* [G, n_rows, 2] or NULL */
  int status;
} select_ctx;

static void select_item(int64_t it, void* p) {
  select_ctx* c = (select_ctx*)p;
  int64_t r = it / c->G;
  int g = (int)(it % c->G);
  int64_t t = c->rows[r];
  double* S = c->S ? c->S + (r * c->G + g) * c->nb : (double*)malloc(sizeof(double) * (size_t)c->nb);
  unsigned char* taken = (unsigned char*)malloc((size_t)c->nb + 1);
  if (!S || !taken) {
    c->status = ORACLE_NO_MEM;
    if (!c->S) free(S);
    free(taken);
    return;
  }
  block_scores_row(c->q_idx_rows + (r * c->G + g) * c->d_I, c->k_idx, t, c->d_I, c->Bk, c->nb, S);
  if (c->blk)
    topk_row(S, t, c->Bk, c->k, c->blk + ((int64_t)g * c->n_rows + r) * c->k,
             c->kth ? c->kth + ((int64_t)g * c->n_rows + r) * 2 : NULL, taken);
  if (!c->S) free(S);
  free(taken);
}

/*
 * Block scores S for the listed query positions (rows[r] = t).
 * q_idx_rows holds the index-query rows of those positions only.
 */
int msa_ref_block_scores(const uint16_t* q_idx_rows, const uint16_t* k_idx, const int64_t* rows,
                         int64_t n_rows, int64_t N, int G, int d_I, int Bk, double* S, int n_threads) {
  if (!q_idx_rows || !k_idx || !rows || !S || N <= 0 || G <= 0 || d_I <= 0 || d_I > 512 || Bk <= 0)
    return ORACLE_BAD_ARG;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return ORACLE_BAD_ARG;
  select_ctx c = {q_idx_rows, k_idx, rows, n_rows, N, (N + Bk - 1) / Bk, G, d_I, Bk, 0, S, NULL, NULL, 0};
  parallel_for(n_rows * G, n_threads, select_item, &c);
  return c.status;
}

/* Selected block sets block_idx[g, r, :] for the listed positions. */
int msa_ref_select_blocks(const uint16_t* q_idx_rows, const uint16_t* k_idx, const int64_t* rows,
                          int64_t n_rows, int64_t N, int G, int d_I, int Bk, int k, int32_t* block_idx,
                          double* kth, int n_threads) {
  if (!q_idx_rows || !k_idx || !rows || !block_idx || N <= 0 || G <= 0 || d_I <= 0 || d_I > 512 || Bk <= 0 ||
      k < 1)
    return ORACLE_BAD_ARG;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return ORACLE_BAD_ARG;
  select_ctx c = {q_idx_rows, k_idx, rows, n_rows, N, (N + Bk - 1) / Bk, G, d_I, Bk, k, NULL, block_idx, kth, 0};
  parallel_for(n_rows * G, n_threads, select_item, &c);
  return c.status;
}

/* ------------------------------------------- FP8 (E4M3) index inputs */
/*
 * [P2] "Co-Design Del Kernel" lists FP8 among the precisions of the pages'
 * kernel, and [P1] 6 "Limitations" 1 notes that the index branch scores the
 * whole context, so the index inputs are the ones worth narrowing.  Reading:
 * q^I and k^I are stored as FP8 E4M3 codes, every product and sum of the
 * scores is exact arithmetic on the decoded values (fp64 here), and the
 * selection rule is unchanged.  A positive factor applied to all of q^I or
 * all of k^I before the cast leaves every row's ordering unchanged, so the
 * selection needs no scale.
 *
 * The encoding is the E4M3 format of the OCP 8-bit floating point
 * specification: sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent field 0 holds the subnormals (m/8) 2^-6; S.1111.111 is NaN; there
 * is no infinity, and the largest finite magnitude is 1.75 * 2^8 = 448.
 */
static double e4m3_to_double(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/*
 * Nearest E4M3 code of the float value v, ties to the even code (round to
 * nearest even), magnitudes past 448 saturated to 448 (there is no
 * infinity to overflow to); NaN gives the positive NaN code 0x7F.
 */
static uint8_t e4m3_from_float(float v) {
  if (isnan(v)) return 0x7F;
  uint8_t s = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (a >= 448.0) return (uint8_t)(s | 0x7E);
  /* spacing of the codes around a: 2^(e-3) in binade [2^e, 2^(e+1)) for
   * e >= -6, and the subnormal spacing 2^-9 below 2^-6 */
  int E;
  frexp(a, &E); /* a = f 2^E with f in [0.5, 1): a lies in binade E-1 */
  int e = E - 1;
  if (a == 0.0 || e < -6) e = -6;
  double q = ldexp(1.0, e - 3);
  double r = rint(a / q) * q; /* a / q is exact; rint rounds half to even */
  if (r == 0.0) return s;
  if (r < ldexp(1.0, -6)) return (uint8_t)(s | (int)(r / ldexp(1.0, -9)));
  frexp(r, &E);
  e = E - 1;
  int m = (int)((r / ldexp(1.0, e) - 1.0) * 8.0);
  return (uint8_t)(s | ((e + 7) << 3) | m);
}

/* Decoded values of n E4M3 codes. */
int msa_ref_e4m3_decode(const uint8_t* codes, int64_t n, double* out) {
  if ((!codes || !out) && n > 0) return ORACLE_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_to_double(codes[i]);
  return ORACLE_OK;
}

/* codes[i] = E4M3 code of the float product (bf16 x[i]) * scale. */
int msa_ref_e4m3_quantize(const uint16_t* x, int64_t n, float scale, uint8_t* codes) {
  if ((!x || !codes) && n > 0) return ORACLE_BAD_ARG;
  for (int64_t i = 0; i < n; ++i) {
    float xf = (float)bf16_to_double(x[i]);
    float p = xf * scale;
    codes[i] = e4m3_from_float(p);
  }
  return ORACLE_OK;
}

/* The 256 decoded values, filled by the exported entry points before any
 * worker thread runs (the same e4m3_to_double values, looked up). */
static double e4m3_value[256];
static void e4m3_fill_values(void) {
  for (int c = 0; c < 256; ++c) e4m3_value[c] = e4m3_to_double((uint8_t)c);
}

/* Step 1 on E4M3 inputs: the same block maxima of the decoded scores. */
static void block_scores_row_e4m3(const uint8_t* qrow, const uint8_t* k_idx, int64_t t, int d_I, int Bk,
                                  int64_t nb, double* S) {
  double inv = 1.0 / sqrt((double)d_I);
  double q[512];
  for (int c = 0; c < d_I; ++c) q[c] = e4m3_value[qrow[c]];
  for (int64_t b = 0; b < nb; ++b) S[b] = -INFINITY;
  for (int64_t j = 0; j <= t; ++j) {
    const uint8_t* kr = k_idx + j * d_I;
    double s = 0.0;
    for (int c = 0; c < d_I; ++c) s += q[c] * e4m3_value[kr[c]];
    s *= inv;
    int64_t b = j / Bk;
    if (s > S[b]) S[b] = s;
  }
}

typedef struct {
  const uint8_t* q_idx_rows; /* [n_rows, G, d_I] E4M3 */
  const uint8_t* k_idx;      /* [N, d_I] E4M3 */
  const int64_t* rows;
  int64_t n_rows, N, nb;
  int G, d_I, Bk, k;
  double* S;
  int32_t* blk;
  double* kth;
  int status;
} select8_ctx;

static void select8_item(int64_t it, void* p) {
  select8_ctx* c = (select8_ctx*)p;
  int64_t r = it / c->G;
  int g = (int)(it % c->G);
  int64_t t = c->rows[r];
  double* S = c->S ? c->S + (r * c->G + g) * c->nb : (double*)malloc(sizeof(double) * (size_t)c->nb);
  unsigned char* taken = (unsigned char*)malloc((size_t)c->nb + 1);
  if (!S || !taken) {
    c->status = ORACLE_NO_MEM;
    if (!c->S) free(S);
    free(taken);
    return;
  }
  block_scores_row_e4m3(c->q_idx_rows + (r * c->G + g) * c->d_I, c->k_idx, t, c->d_I, c->Bk, c->nb, S);
  if (c->blk)
    topk_row(S, t, c->Bk, c->k, c->blk + ((int64_t)g * c->n_rows + r) * c->k,
             c->kth ? c->kth + ((int64_t)g * c->n_rows + r) * 2 : NULL, taken);
  if (!c->S) free(S);
  free(taken);
}

/* msa_ref_block_scores on E4M3 codes. */
int msa_ref_block_scores_e4m3(const uint8_t* q_idx_rows, const uint8_t* k_idx, const int64_t* rows,
                              int64_t n_rows, int64_t N, int G, int d_I, int Bk, double* S, int n_threads) {
  if (!q_idx_rows || !k_idx || !rows || !S || N <= 0 || G <= 0 || d_I <= 0 || d_I > 512 || Bk <= 0)
    return ORACLE_BAD_ARG;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return ORACLE_BAD_ARG;
  select8_ctx c = {q_idx_rows, k_idx, rows, n_rows, N, (N + Bk - 1) / Bk, G, d_I, Bk, 0, S, NULL, NULL, 0};
  e4m3_fill_values();
  parallel_for(n_rows * G, n_threads, select8_item, &c);
  return c.status;
}

/* msa_ref_select_blocks on E4M3 codes. */
int msa_ref_select_blocks_e4m3(const uint8_t* q_idx_rows, const uint8_t* k_idx, const int64_t* rows,
                               int64_t n_rows, int64_t N, int G, int d_I, int Bk, int k, int32_t* block_idx,
                               double* kth, int n_threads) {
  if (!q_idx_rows || !k_idx || !rows || !block_idx || N <= 0 || G <= 0 || d_I <= 0 || d_I > 512 || Bk <= 0 ||
      k < 1)
    return ORACLE_BAD_ARG;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return ORACLE_BAD_ARG;
  select8_ctx c = {q_idx_rows, k_idx, rows, n_rows, N, (N + Bk - 1) / Bk, G, d_I, Bk, k, NULL, block_idx, kth, 0};
  e4m3_fill_values();
  parallel_for(n_rows * G, n_threads, select8_item, &c);
  return c.status;
}

/* ----------------------------------------------- step 3: B -> B* inversion */
/*
 * [P4] "バックワードパス": B[g, t, slot] -> block becomes B*[g, block] -> the
 * (t, slot) pairs that chose it.  CSR per group: entries of block b are
 * entries[g*N*k + row_ptr[g*(nb+1) + b] ...], each t*k + slot, ascending t.
 * Ids outside [0, nb) and -1 are not listed.
 */
int msa_ref_invert_blocks(const int32_t* block_idx, int64_t N, int G, int Bk, int k, int32_t* row_ptr,
                          int32_t* entries, int32_t* n_entries) {
  if (!block_idx || !row_ptr || !entries || !n_entries || N <= 0 || G <= 0 || Bk <= 0 || k < 1)
    return ORACLE_BAD_ARG;
  int64_t nb = (N + Bk - 1) / Bk;
  for (int g = 0; g < G; ++g) {
    const int32_t* B = block_idx + (int64_t)g * N * k;
    int32_t* rp = row_ptr + (int64_t)g * (nb + 1);
    int32_t* E = entries + (int64_t)g * N * k;
    for (int64_t b = 0; b <= nb; ++b) rp[b] = 0;
    for (int64_t e = 0; e < N * k; ++e)
      if (B[e] >= 0 && B[e] < nb) rp[B[e] + 1] += 1;
    for (int64_t b = 0; b < nb; ++b) rp[b + 1] += rp[b];
    n_entries[g] = rp[nb];
    /* fill each block's list by scanning (t, slot) in increasing order */
    int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nb + 1));
    if (!cursor) return ORACLE_NO_MEM;
    for (int64_t b = 0; b < nb; ++b) cursor[b] = rp[b];
    for (int64_t e = 0; e < N * k; ++e) {
      int32_t b = B[e];
      if (b >= 0 && b < nb) E[cursor[b]++] = (int32_t)e;
    }
    free(cursor);
  }
  return ORACLE_OK;
}

/* --------------------------------------- step 4: attention over a key set */
/*
 * [P1] 1-1 and 3-3: out = softmax(scale * q K_J^T) V_J over the key set J,
 * lse = log sum_j exp(scale q.k_j) ([P1] 3-5 item 4, [P4] main LSE).
 * An empty J gives out = 0 and lse = -inf.
 */
static void attend_set(const uint16_t* q /*[d]*/, const uint16_t* K, const uint16_t* V, int64_t kv_stride,
                       const int64_t* J, int64_t nJ, int d, double scale, double* out, double* lse,
                       double* z /*[nJ] scratch*/) {
  for (int c = 0; c < d; ++c) out[c] = 0.0;
  if (nJ == 0) {
    *lse = -INFINITY;
    return;
  }
  double m = -INFINITY;
  for (int64_t i = 0; i < nJ; ++i) {
    z[i] = scale * dot_bf16(q, K + J[i] * kv_stride, d);
    if (z[i] > m) m = z[i];
  }
  double l = 0.0;
  for (int64_t i = 0; i < nJ; ++i) {
    double p = exp(z[i] - m);
    l += p;
    const uint16_t* vr = V + J[i] * kv_stride;
    for (int c = 0; c < d; ++c) out[c] += p * bf16_to_double(vr[c]);
  }
  for (int c = 0; c < d; ++c) out[c] /= l;
  *lse = m + log(l);
}

/*
 * J(t, set) = { j : floor(j / Bk) is an id of the set, j <= t } in slot order,
 * ascending j within a block ([P1] 2-3 and 3-3; [P2] "causally visible").
 * A repeated id counts once.
 */
static int64_t key_set(const int32_t* sel, int k, int64_t t, int Bk, int64_t nb, int64_t* J) {
  int64_t n = 0;
  for (int s = 0; s < k; ++s) {
    int32_t b = sel[s];
    if (b < 0 || b >= nb) continue;
    int dup = 0;
    for (int s2 = 0; s2 < s; ++s2)
      if (sel[s2] == b) dup = 1;
    if (dup) continue;
    for (int64_t j = (int64_t)b * Bk; j < (int64_t)(b + 1) * Bk && j <= t; ++j) J[n++] = j;
  }
  return n;
}

typedef struct {
  const uint16_t *q_rows, *K, *V;
  const int32_t* blk; /* [G, n_rows, k] or NULL for dense */
  const int64_t* rows;
  int64_t n_rows, N, nb;
  int H_q, H_kv, d, Bk, k;
  double scale;
  double *out, *lse;
  int status;
} attn_ctx;

static void attn_item(int64_t it, void* p) {
  attn_ctx* c = (attn_ctx*)p;
  int64_t r = it / c->H_q;
  int h = (int)(it % c->H_q);
  int g = h / (c->H_q / c->H_kv); /* [P1] 1-1: head h reads the K/V of its GQA group */
  int64_t t = c->rows[r];
  int64_t cap = c->blk ? (int64_t)c->k * c->Bk : t + 1;
  int64_t* J = (int64_t*)malloc(sizeof(int64_t) * (size_t)(cap + 1));
  double* z = (double*)malloc(sizeof(double) * (size_t)(cap + 1));
  if (!J || !z) {
    c->status = ORACLE_NO_MEM;
    free(J);
    free(z);
    return;
  }
  int64_t nJ;
  if (c->blk) {
    nJ = key_set(c->blk + ((int64_t)g * c->n_rows + r) * c->k, c->k, t, c->Bk, c->nb, J);
  } else {
    nJ = t + 1; /* dense causal: every j <= t */
    for (int64_t j = 0; j <= t; ++j) J[j] = j;
  }
  int64_t kv_stride = (int64_t)c->H_kv * c->d;
  attend_set(c->q_rows + (r * c->H_q + h) * c->d, c->K + (int64_t)g * c->d, c->V + (int64_t)g * c->d,
             kv_stride, J, nJ, c->d, c->scale, c->out + (r * c->H_q + h) * c->d, c->lse + r * c->H_q + h, z);
  free(J);
  free(z);
}

/*
 * Block-sparse attention of the listed positions over a given selection
 * (block_idx_rows[g, r, :] is the set of row r).  q_rows: [n_rows, H_q, d];
 * K, V: [N, H_kv, d].  out: [n_rows, H_q, d], lse: [n_rows, H_q].
 */
int msa_ref_sparse_attn(const uint16_t* q_rows, const uint16_t* K, const uint16_t* V,
                        const int32_t* block_idx_rows, const int64_t* rows, int64_t n_rows, int64_t N,
                        int H_q, int H_kv, int d, int Bk, int k, double scale, double* out, double* lse,
                        int n_threads) {
  if (!q_rows || !K || !V || !block_idx_rows || !rows || !out || !lse || N <= 0 || H_kv <= 0 ||
      H_q % H_kv != 0 || d <= 0 || Bk <= 0 || k < 1)
    return ORACLE_BAD_ARG;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return ORACLE_BAD_ARG;
  attn_ctx c = {q_rows, K, V, block_idx_rows, rows, n_rows, N, (N + Bk - 1) / Bk, H_q, H_kv, d, Bk, k,
                scale, out, lse, 0};
  parallel_for(n_rows * H_q, n_threads, attn_item, &c);
  return c.status;
}

/* Dense causal GQA attention ([P1] 1-1) of the listed positions. */
int msa_ref_dense_attn(const uint16_t* q_rows, const uint16_t* K, const uint16_t* V, const int64_t* rows,
                       int64_t n_rows, int64_t N, int H_q, int H_kv, int d, double scale, double* out,
                       double* lse, int n_threads) {
  if (!q_rows || !K || !V || !rows || !out || !lse || N <= 0 || H_kv <= 0 || H_q % H_kv != 0 || d <= 0)
    return ORACLE_BAD_ARG;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return ORACLE_BAD_ARG;
  attn_ctx c = {q_rows, K, V, NULL, rows, n_rows, N, 1, H_q, H_kv, d, 1, 1, scale, out, lse, 0};
  parallel_for(n_rows * H_q, n_threads, attn_item, &c);
  return c.status;
}

/* ------------------------------------------------------- step 6: decode */
typedef struct {
  const uint16_t *q_t, *q_idx_t, *k_idx_cache, *k_cache, *v_cache;
  const int64_t* ctx_len;
  int64_t ctx_max, nb_max;
  int B, H_q, H_kv, d, d_I, Bk, k;
  double scale;
  double *out, *lse, *kth;
  int32_t* blk; /* [B, G, k] */
  int status;
} decode_ctx;

static void decode_select_item(int64_t it, void* p) {
  decode_ctx* c = (decode_ctx*)p;
  int G = c->H_kv;
  int64_t b = it / G;
  int g = (int)(it % G);
  int64_t t = c->ctx_len[b] - 1;
  int64_t nb = t / c->Bk + 1;
  double* S = (double*)malloc(sizeof(double) * (size_t)nb);
  unsigned char* taken = (unsigned char*)malloc((size_t)nb + 1);
  if (!S || !taken) {
    c->status = ORACLE_NO_MEM;
    free(S);
    free(taken);
    return;
  }
  block_scores_row(c->q_idx_t + (b * G + g) * c->d_I, c->k_idx_cache + b * c->ctx_max * c->d_I, t, c->d_I,
                   c->Bk, nb, S);
  topk_row(S, t, c->Bk, c->k, c->blk + (b * G + g) * c->k, c->kth ? c->kth + (b * G + g) * 2 : NULL, taken);
  free(S);
  free(taken);
}

static void decode_attn_item(int64_t it, void* p) {
  decode_ctx* c = (decode_ctx*)p;
  int64_t b = it / c->H_q;
  int h = (int)(it % c->H_q);
  int G = c->H_kv;
  int g = h / (c->H_q / G);
  int64_t t = c->ctx_len[b] - 1;
  int64_t* J = (int64_t*)malloc(sizeof(int64_t) * (size_t)c->k * c->Bk);
  double* z = (double*)malloc(sizeof(double) * (size_t)c->k * c->Bk);
  if (!J || !z) {
    c->status = ORACLE_NO_MEM;
    free(J);
    free(z);
    return;
  }
  int64_t nJ = key_set(c->blk + (b * G + g) * c->k, c->k, t, c->Bk, c->nb_max, J);
  int64_t kv_stride = (int64_t)G * c->d;
  const uint16_t* K = c->k_cache + b * c->ctx_max * kv_stride + (int64_t)g * c->d;
  const uint16_t* V = c->v_cache + b * c->ctx_max * kv_stride + (int64_t)g * c->d;
  attend_set(c->q_t + (b * c->H_q + h) * c->d, K, V, kv_stride, J, nJ, c->d, c->scale,
             c->out + (b * c->H_q + h) * c->d, c->lse + b * c->H_q + h, z);
  free(J);
  free(z);
}

/*
 * One decode step ([P3] section 2): per sequence b the query at
 * t = ctx_len[b] - 1 scores the whole index-key cache, keeps its block set
 * (steps 1-2) and attends over the selected blocks' tokens j <= t (step 4).
 * q_t [B,H_q,d], q_idx_t [B,G,d_I], k_idx_cache [B,ctx_max,d_I],
 * k_cache / v_cache [B,ctx_max,H_kv,d].  Outputs out [B,H_q,d], lse [B,H_q],
 * block_idx [B,G,k], kth [B,G,2] (nullable).
 */
int msa_ref_decode(const uint16_t* q_t, const uint16_t* q_idx_t, const uint16_t* k_idx_cache,
                   const uint16_t* k_cache, const uint16_t* v_cache, const int64_t* ctx_len, int B,
                   int64_t ctx_max, int H_q, int H_kv, int d, int d_I, int Bk, int k, double scale,
                   double* out, double* lse, int32_t* block_idx, double* kth, int n_threads) {
  if (!q_t || !q_idx_t || !k_idx_cache || !k_cache || !v_cache || !ctx_len || !out || !lse || !block_idx ||
      B <= 0 || ctx_max <= 0 || H_kv <= 0 || H_q % H_kv != 0 || d <= 0 || d_I <= 0 || d_I > 512 || Bk <= 0 ||
      k < 1)
    return ORACLE_BAD_ARG;
  for (int b = 0; b < B; ++b)
    if (ctx_len[b] < 1 || ctx_len[b] > ctx_max) return ORACLE_BAD_ARG;
  decode_ctx c = {q_t, q_idx_t, k_idx_cache, k_cache, v_cache, ctx_len, ctx_max, (ctx_max + Bk - 1) / Bk,
                  B, H_q, H_kv, d, d_I, Bk, k, scale, out, lse, kth, block_idx, 0};
  parallel_for((int64_t)B * H_kv, n_threads, decode_select_item, &c);
  if (c.status) return c.status;
  parallel_for((int64_t)B * H_q, n_threads, decode_attn_item, &c);
  return c.status;
}


/* ------------------------------------------------------------- backward */
/*
 * One row (t, g) of the backward, for every head h of group g:
 *   forward, recomputed: z_j = scale q_{t,h}.k_{j,g}, P_j = exp(z_j - lse),
 *   O = sum_j P_j v_{j,g} ([P1] 3-3);
 *   main gradient of a softmax attention with upstream dO:
 *     D = dO.O, dP_j = dO.v_j, dZ_j = P_j (dP_j - D),
 *     dq_{t,h} = scale sum_j dZ_j k_j, dk_j += scale dZ_j q_{t,h}, dv_j += P_j dO;
 *   index branch ([P1] 4-2, 4-3; [P4] KL section): teacher pbar_j = mean_h P_j
 *   (detached), index logits zI_j = q^I.k^I_j / sqrt(d_I), pI = softmax_J(zI),
 *     KL = sum_j pbar_j (log pbar_j - log pI_j),
 *     dL/dzI_j = w (pI_j - pbar_j),
 *     dq^I_{t,g} = sum_j dL/dzI_j k^I_j / sqrt(d_I), dk^I_j += dL/dzI_j q^I_{t,g} / sqrt(d_I).
 * Sums over (t, h) into dk, dv and dk^I go to the work item's private
 * accumulators (dk_acc/dv_acc [N][d] of group g, dkI_acc [N][d_I]).
 */
typedef struct {
  const uint16_t *q, *K, *V, *q_idx, *k_idx, *dO;
  const int32_t* blk;
  const int64_t* rows; /* NULL: every position; else only these (dq, dq_idx and kl rows only) */
  int64_t n_rows;
  int64_t N, nb;
  int H_q, H_kv, d, d_I, Bk, k, chunks;
  double scale, kl_weight;
  double *dq, *dq_idx, *kl;          /* row-local outputs */
  double *dk_acc, *dv_acc, *dkI_acc; /* [items][N][d], [items][N][d], [items][N][d_I] */
  int status;
} bwd_ctx;

static void bwd_item(int64_t it, void* p) {
  bwd_ctx* c = (bwd_ctx*)p;
  const int g = (int)(it / c->chunks), ch = (int)(it % c->chunks);
  const int gs = c->H_q / c->H_kv, d = c->d, dI = c->d_I;
  const int64_t r0 = c->n_rows * ch / c->chunks, r1 = c->n_rows * (ch + 1) / c->chunks;
  const int64_t cap = (int64_t)c->k * c->Bk;
  const int64_t kv_stride = (int64_t)c->H_kv * d;
  double* dk_acc = c->dk_acc ? c->dk_acc + it * c->N * d : NULL;
  double* dv_acc = c->dv_acc ? c->dv_acc + it * c->N * d : NULL;
  double* dkI_acc = c->dkI_acc ? c->dkI_acc + it * c->N * dI : NULL;
  int64_t* J = (int64_t*)malloc(sizeof(int64_t) * (size_t)cap);
  double* P = (double*)malloc(sizeof(double) * (size_t)(cap * gs));
  double* pbar = (double*)malloc(sizeof(double) * (size_t)cap);
  double* zI = (double*)malloc(sizeof(double) * (size_t)cap);
  double* O = (double*)malloc(sizeof(double) * (size_t)d);
  if (!J || !P || !pbar || !zI || !O) {
    c->status = ORACLE_NO_MEM;
    free(J), free(P), free(pbar), free(zI), free(O);
    return;
  }
  for (int64_t ri = r0; ri < r1; ++ri) {
    const int64_t t = c->rows ? c->rows[ri] : ri;
    const int64_t nJ = key_set(c->blk + ((int64_t)g * c->N + t) * c->k, c->k, t, c->Bk, c->nb, J);
    for (int64_t i = 0; i < nJ; ++i) pbar[i] = 0.0;
    for (int hh = 0; hh < gs; ++hh) {
      const int h = g * gs + hh;
      const uint16_t* qr = c->q + (t * c->H_q + h) * d;
      const uint16_t* dOr = c->dO + (t * c->H_q + h) * d;
      double* Ph = P + (int64_t)hh * cap;
      double* dq = c->dq + (t * c->H_q + h) * d;
      for (int x = 0; x < d; ++x) dq[x] = 0.0;
      if (nJ == 0) continue;
      double m = -INFINITY;
      for (int64_t i = 0; i < nJ; ++i) {
        Ph[i] = c->scale * dot_bf16(qr, c->K + J[i] * kv_stride + (int64_t)g * d, d);
        if (Ph[i] > m) m = Ph[i];
      }
      double l = 0.0;
      for (int64_t i = 0; i < nJ; ++i) l += exp(Ph[i] - m);
      const double lse = m + log(l);
      for (int x = 0; x < d; ++x) O[x] = 0.0;
      for (int64_t i = 0; i < nJ; ++i) {
        Ph[i] = exp(Ph[i] - lse);
        const uint16_t* vr = c->V + J[i] * kv_stride + (int64_t)g * d;
        for (int x = 0; x < d; ++x) O[x] += Ph[i] * bf16_to_double(vr[x]);
      }
      double D = 0.0;
      for (int x = 0; x < d; ++x) D += bf16_to_double(dOr[x]) * O[x];
      for (int64_t i = 0; i < nJ; ++i) {
        const uint16_t* kr = c->K + J[i] * kv_stride + (int64_t)g * d;
        const uint16_t* vr = c->V + J[i] * kv_stride + (int64_t)g * d;
        const double dZ = Ph[i] * (dot_bf16(dOr, vr, d) - D);
        for (int x = 0; x < d; ++x) dq[x] += c->scale * dZ * bf16_to_double(kr[x]);
        if (dk_acc) {
          double* dkr = dk_acc + J[i] * d;
          double* dvr = dv_acc + J[i] * d;
          for (int x = 0; x < d; ++x) {
            dkr[x] += c->scale * dZ * bf16_to_double(qr[x]);
            dvr[x] += Ph[i] * bf16_to_double(dOr[x]);
          }
        }
        pbar[i] += Ph[i] / gs;
      }
    }
    /* index branch */
    const uint16_t* qIr = c->q_idx + (t * c->H_kv + g) * dI;
    double* dqI = c->dq_idx + (t * c->H_kv + g) * dI;
    for (int x = 0; x < dI; ++x) dqI[x] = 0.0;
    double* klr = c->kl + (int64_t)g * c->N + t;
    *klr = 0.0;
    if (nJ == 0) continue;
    const double sI = 1.0 / sqrt((double)dI);
    double mI = -INFINITY;
    for (int64_t i = 0; i < nJ; ++i) {
      zI[i] = sI * dot_bf16(qIr, c->k_idx + J[i] * dI, dI);
      if (zI[i] > mI) mI = zI[i];
    }
    double lI = 0.0;
    for (int64_t i = 0; i < nJ; ++i) lI += exp(zI[i] - mI);
    const double lseI = mI + log(lI);
    double kl = 0.0;
    for (int64_t i = 0; i < nJ; ++i) {
      const double logpI = zI[i] - lseI;
      const double pI = exp(logpI);
      if (pbar[i] > 0.0) kl += pbar[i] * (log(pbar[i]) - logpI);
      const double dz = c->kl_weight * (pI - pbar[i]);
      const uint16_t* kIr = c->k_idx + J[i] * dI;
      for (int x = 0; x < dI; ++x) dqI[x] += sI * dz * bf16_to_double(kIr[x]);
      if (dkI_acc) {
        double* dkIr = dkI_acc + J[i] * dI;
        for (int x = 0; x < dI; ++x) dkIr[x] += sI * dz * bf16_to_double(qIr[x]);
      }
    }
    *klr = kl;
  }
  free(J), free(P), free(pbar), free(zI), free(O);
}

/*
 * Backward of block-sparse attention and of the index branch's KL loss for
 * all N positions.  q, dO: [N, H_q, d]; K, V: [N, H_kv, d]; q_idx: [N, G,
 * d_I]; k_idx: [N, d_I]; block_idx: [G, N, k].  Outputs (double): dq [N,
 * H_q, d], dk and dv [N, H_kv, d], dq_idx [N, G, d_I], dk_idx [N, d_I], kl
 * [G, N] (each row's KL(teacher || index)).
 */
int msa_ref_sparse_attn_bwd(const uint16_t* q, const uint16_t* K, const uint16_t* V, const uint16_t* q_idx,
                            const uint16_t* k_idx, const int32_t* block_idx, const uint16_t* dO, int64_t N, int H_q,
                            int H_kv, int d, int d_I, int Bk, int k, double scale, double kl_weight, double* dq,
                            double* dk, double* dv, double* dq_idx, double* dk_idx, double* kl, int n_threads) {
  if (!q || !K || !V || !q_idx || !k_idx || !block_idx || !dO || !dq || !dk || !dv || !dq_idx || !dk_idx || !kl ||
      N <= 0 || H_kv <= 0 || H_q % H_kv != 0 || d <= 0 || d_I <= 0 || Bk <= 0 || k < 1)
    return ORACLE_BAD_ARG;
  int chunks = n_threads / H_kv;
  if (chunks < 1) chunks = 1;
  const double acc_bytes = (double)N * (2 * d + d_I) * 8.0;
  while (chunks > 1 && acc_bytes * chunks * H_kv > 2.0e9) --chunks;
  const int64_t items = (int64_t)H_kv * chunks;
  double* dk_acc = (double*)calloc((size_t)(items * N * d), sizeof(double));
  double* dv_acc = (double*)calloc((size_t)(items * N * d), sizeof(double));
  double* dkI_acc = (double*)calloc((size_t)(items * N * d_I), sizeof(double));
  if (!dk_acc || !dv_acc || !dkI_acc) {
    free(dk_acc), free(dv_acc), free(dkI_acc);
    return ORACLE_NO_MEM;
  }
  bwd_ctx c = {q, K, V, q_idx, k_idx, dO, block_idx, NULL, N, N, (N + Bk - 1) / Bk, H_q, H_kv, d, d_I, Bk, k,
               chunks, scale, kl_weight, dq, dq_idx, kl, dk_acc, dv_acc, dkI_acc, 0};
  parallel_for(items, n_threads, bwd_item, &c);
  /* sum the items' accumulators */
  for (int64_t j = 0; j < N; ++j) {
    for (int g = 0; g < H_kv; ++g)
      for (int x = 0; x < d; ++x) {
        double a = 0.0, b = 0.0;
        for (int ch = 0; ch < chunks; ++ch) {
          const int64_t itm = (int64_t)g * chunks + ch;
          a += dk_acc[(itm * N + j) * d + x];
          b += dv_acc[(itm * N + j) * d + x];
        }
        dk[(j * H_kv + g) * d + x] = a;
        dv[(j * H_kv + g) * d + x] = b;
      }
    for (int x = 0; x < d_I; ++x) {
      double a = 0.0;
      for (int64_t itm = 0; itm < items; ++itm) a += dkI_acc[(itm * N + j) * d_I + x];
      dk_idx[j * d_I + x] = a;
    }
  }
  free(dk_acc), free(dv_acc), free(dkI_acc);
  return c.status;
}

/*
 * The row-local part of the backward (dq, dq_idx and kl) for the listed
 * positions only, over the full-size inputs: dq [n_rows, H_q, d], dq_idx
 * [n_rows, G, d_I], kl [G, n_rows] in list order.  Same arithmetic as
 * msa_ref_sparse_attn_bwd for those rows.
 */
int msa_ref_sparse_attn_bwd_rows(const uint16_t* q, const uint16_t* K, const uint16_t* V, const uint16_t* q_idx,
                                 const uint16_t* k_idx, const int32_t* block_idx, const uint16_t* dO,
                                 const int64_t* rows, int64_t n_rows, int64_t N, int H_q, int H_kv, int d, int d_I,
                                 int Bk, int k, double scale, double kl_weight, double* dq_rows, double* dq_idx_rows,
                                 double* kl_rows, int n_threads) {
  if (!q || !K || !V || !q_idx || !k_idx || !block_idx || !dO || !rows || !dq_rows || !dq_idx_rows || !kl_rows ||
      n_rows <= 0 || N <= 0 || H_kv <= 0 || H_q % H_kv != 0 || d <= 0 || d_I <= 0 || Bk <= 0 || k < 1)
    return ORACLE_BAD_ARG;
  for (int64_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= N) return ORACLE_BAD_ARG;
  /* full-size row outputs, only the listed rows written; copied out in list order */
  double* dq = (double*)calloc((size_t)(N * H_q * d), sizeof(double));
  double* dqI = (double*)calloc((size_t)(N * H_kv * d_I), sizeof(double));
  double* kl = (double*)calloc((size_t)(H_kv * N), sizeof(double));
  if (!dq || !dqI || !kl) {
    free(dq), free(dqI), free(kl);
    return ORACLE_NO_MEM;
  }
  int chunks = n_threads / H_kv;
  if (chunks < 1) chunks = 1;
  bwd_ctx c = {q, K, V, q_idx, k_idx, dO, block_idx, rows, n_rows, N, (N + Bk - 1) / Bk, H_q, H_kv, d, d_I, Bk, k,
               chunks, scale, kl_weight, dq, dqI, kl, NULL, NULL, NULL, 0};
  parallel_for((int64_t)H_kv * chunks, n_threads, bwd_item, &c);
  for (int64_t r = 0; r < n_rows; ++r) {
    const int64_t t = rows[r];
    memcpy(dq_rows + r * H_q * d, dq + t * H_q * d, sizeof(double) * (size_t)(H_q * d));
    memcpy(dq_idx_rows + r * H_kv * d_I, dqI + t * H_kv * d_I, sizeof(double) * (size_t)(H_kv * d_I));
    for (int g = 0; g < H_kv; ++g) kl_rows[(int64_t)g * n_rows + r] = kl[(int64_t)g * N + t];
  }
  free(dq), free(dqI), free(kl);
  return c.status;
}


/* -------------------------------------------------------------- warmup mode */
/*
 * [P1] 4-4 "Indexer warmup": before top-k routing is switched on, the main
 * branch runs full (dense causal) attention and the index branch learns the KL
 * alignment against the full-context teacher.  Per row (t, g), over every
 * j <= t:
 *   z_{h,j} = scale q_{t,h}.k_{j,g}, P_{h,j} = exp(z_{h,j} - lse_h) for the
 *   group's heads h ([P1] 1-1, dense causal GQA); teacher pbar_j = mean_h P_{h,j}
 *   ([P1] 4-2, detached); index logits zI_j = q^I.k^I_j / sqrt(d_I);
 *   KL = sum_j pbar_j (log pbar_j - log pI_j) with pI = softmax_j(zI);
 *   dL/dzI_j = w (pI_j - pbar_j) ([P4] KL section);
 *   dq^I_{t,g} = sum_j dL/dzI_j k^I_j / sqrt(d_I),
 *   dk^I_j += dL/dzI_j q^I_{t,g} / sqrt(d_I).
 * The main branch's own output is msa_ref_dense_attn.
 */
typedef struct {
  const uint16_t *q, *K, *q_idx, *k_idx;
  const int64_t* rows; /* NULL: every position */
  int64_t n_rows, N;
  int H_q, H_kv, d, d_I, chunks;
  double scale, kl_weight;
  double *kl, *dq_idx; /* [G, n_rows], [n_rows, G, d_I] */
  double* lse_idx;     /* [G, n_rows] or NULL: the index branch's lse per row */
  double* dkI_acc;     /* [items][N][d_I] or NULL */
  int status;
} warm_ctx;

static void warm_item(int64_t it, void* p) {
  warm_ctx* c = (warm_ctx*)p;
  const int g = (int)(it / c->chunks), ch = (int)(it % c->chunks);
  const int gs = c->H_q / c->H_kv, d = c->d, dI = c->d_I;
  const int64_t r0 = c->n_rows * ch / c->chunks, r1 = c->n_rows * (ch + 1) / c->chunks;
  const int64_t kv_stride = (int64_t)c->H_kv * d;
  double* dkI_acc = c->dkI_acc ? c->dkI_acc + it * c->N * dI : NULL;
  double* z = (double*)malloc(sizeof(double) * (size_t)c->N);
  double* pbar = (double*)malloc(sizeof(double) * (size_t)c->N);
  if (!z || !pbar) {
    c->status = ORACLE_NO_MEM;
    free(z), free(pbar);
    return;
  }
  const double sI = 1.0 / sqrt((double)dI);
  for (int64_t ri = r0; ri < r1; ++ri) {
    const int64_t t = c->rows ? c->rows[ri] : ri;
    const int64_t n = t + 1; /* keys 0..t */
    for (int64_t j = 0; j < n; ++j) pbar[j] = 0.0;
    for (int hh = 0; hh < gs; ++hh) {
      const uint16_t* qr = c->q + (t * c->H_q + g * gs + hh) * d;
      double m = -INFINITY;
      for (int64_t j = 0; j < n; ++j) {
        z[j] = c->scale * dot_bf16(qr, c->K + j * kv_stride + (int64_t)g * d, d);
        if (z[j] > m) m = z[j];
      }
      double l = 0.0;
      for (int64_t j = 0; j < n; ++j) l += exp(z[j] - m);
      const double lse = m + log(l);
      for (int64_t j = 0; j < n; ++j) pbar[j] += exp(z[j] - lse) / gs;
    }
    const uint16_t* qIr = c->q_idx + (t * c->H_kv + g) * dI;
    double mI = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
      z[j] = sI * dot_bf16(qIr, c->k_idx + j * dI, dI);
      if (z[j] > mI) mI = z[j];
    }
    double lI = 0.0;
    for (int64_t j = 0; j < n; ++j) lI += exp(z[j] - mI);
    const double lseI = mI + log(lI);
    if (c->lse_idx) c->lse_idx[(int64_t)g * c->n_rows + ri] = lseI;
    double* dqI = c->dq_idx + (ri * c->H_kv + g) * dI;
    for (int x = 0; x < dI; ++x) dqI[x] = 0.0;
    double kl = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      const double logpI = z[j] - lseI;
      if (pbar[j] > 0.0) kl += pbar[j] * (log(pbar[j]) - logpI);
      const double dz = c->kl_weight * (exp(logpI) - pbar[j]);
      const uint16_t* kIr = c->k_idx + j * dI;
      for (int x = 0; x < dI; ++x) dqI[x] += sI * dz * bf16_to_double(kIr[x]);
      if (dkI_acc) {
        double* dkIr = dkI_acc + j * dI;
        for (int x = 0; x < dI; ++x) dkIr[x] += sI * dz * bf16_to_double(qIr[x]);
      }
    }
    c->kl[(int64_t)g * c->n_rows + ri] = kl;
  }
  free(z), free(pbar);
}

/*
 * Warmup mode's index-branch loss and gradients.  rows == NULL: every
 * position (n_rows = N), and dk_idx [N, d_I] is written; otherwise only the
 * listed positions' kl [G, n_rows] and dq_idx [n_rows, G, d_I] (dk_idx may be
 * NULL).  lse_idx [G, n_rows] (nullable): each row's index log-sum-exp.
 * q [N, H_q, d], K [N, H_kv, d], q_idx [N, G, d_I], k_idx [N, d_I].
 */
int msa_ref_warmup_index(const uint16_t* q, const uint16_t* K, const uint16_t* q_idx, const uint16_t* k_idx,
                         const int64_t* rows, int64_t n_rows, int64_t N, int H_q, int H_kv, int d, int d_I,
                         double scale, double kl_weight, double* kl, double* dq_idx, double* dk_idx,
                         double* lse_idx, int n_threads) {
  if (!q || !K || !q_idx || !k_idx || !kl || !dq_idx || N <= 0 || H_kv <= 0 || H_q % H_kv != 0 || d <= 0 ||
      d_I <= 0 || (!rows && (n_rows != N || !dk_idx)))
    return ORACLE_BAD_ARG;
  if (rows)
    for (int64_t r = 0; r < n_rows; ++r)
      if (rows[r] < 0 || rows[r] >= N) return ORACLE_BAD_ARG;
  int chunks = n_threads / H_kv;
  if (chunks < 1) chunks = 1;
  const int want_dk = rows == NULL;
  while (want_dk && chunks > 1 && (double)N * d_I * 8.0 * chunks * H_kv > 2.0e9) --chunks;
  const int64_t items = (int64_t)H_kv * chunks;
  double* dkI_acc = want_dk ? (double*)calloc((size_t)(items * N * d_I), sizeof(double)) : NULL;
  if (want_dk && !dkI_acc) return ORACLE_NO_MEM;
  warm_ctx c = {q, K, q_idx, k_idx, rows, n_rows, N, H_q, H_kv, d, d_I, chunks, scale, kl_weight, kl, dq_idx,
                lse_idx, dkI_acc, 0};
  parallel_for(items, n_threads, warm_item, &c);
  if (want_dk) {
    for (int64_t j = 0; j < N; ++j)
      for (int x = 0; x < d_I; ++x) {
        double a = 0.0;
        for (int64_t itm = 0; itm < items; ++itm) a += dkI_acc[(itm * N + j) * d_I + x];
        dk_idx[j * d_I + x] = a;
      }
    free(dkI_acc);
  }
  return c.status;
}
