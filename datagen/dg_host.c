/*
 * Host (CPU) fill routines of the seeded synthetic-input generator.
 * Bit-identical to the device routines in dg_cuda.cu (same dg_core.h).
 * Holds none of the sparse-attention method's arithmetic.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#include "dg_core.h"

typedef struct {
  int64_t lo, hi;
  void* ctx;
  void (*fn)(int64_t lo, int64_t hi, void* ctx);
} dg_range_t;

static void* dg_range_main(void* p) {
  dg_range_t* r = (dg_range_t*)p;
  r->fn(r->lo, r->hi, r->ctx);
  return NULL;
}

static void dg_parallel(int64_t n, int n_threads, void (*fn)(int64_t, int64_t, void*), void* ctx) {
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  if ((int64_t)n_threads > n) n_threads = (int)(n > 0 ? n : 1);
  pthread_t th[256];
  dg_range_t rg[256];
  for (int i = 0; i < n_threads; ++i) {
    rg[i].lo = n * i / n_threads;
    rg[i].hi = n * (i + 1) / n_threads;
    rg[i].ctx = ctx;
    rg[i].fn = fn;
  }
  for (int i = 1; i < n_threads; ++i) pthread_create(&th[i], NULL, dg_range_main, &rg[i]);
  dg_range_main(&rg[0]);
  for (int i = 1; i < n_threads; ++i) pthread_join(th[i], NULL);
}

/* ---- plain normal fill: out[i] = bf16(normal(first + i)) ---------------- */
typedef struct {
  uint16_t* out;
  uint64_t key;
  int64_t first;
} dg_fill_ctx;

static void dg_fill_body(int64_t lo, int64_t hi, void* p) {
  dg_fill_ctx* c = (dg_fill_ctx*)p;
  for (int64_t i = lo; i < hi; ++i)
    c->out[i] = dg_bf16_rne(dg_normal(c->key, (uint64_t)(c->first + i)));
}

void dg_host_fill_normal(uint16_t* out, int64_t n, uint64_t seed, uint32_t tensor_id, int64_t first,
                         int n_threads) {
  dg_fill_ctx c = {out, dg_stream_key(seed, tensor_id), first};
  dg_parallel(n, n_threads, dg_fill_body, &c);
}

/* ---- selected rows: out[r, :] = bf16(normal(row_ids[r] * row_len + c)) ---- */
typedef struct {
  uint16_t* out;
  uint64_t key;
  const int64_t* row_ids;
  int64_t row_len;
} dg_rows_ctx;

static void dg_rows_body(int64_t lo, int64_t hi, void* p) {
  dg_rows_ctx* c = (dg_rows_ctx*)p;
  for (int64_t r = lo; r < hi; ++r) {
    uint64_t base = (uint64_t)c->row_ids[r] * (uint64_t)c->row_len;
    for (int64_t j = 0; j < c->row_len; ++j)
      c->out[r * c->row_len + j] = dg_bf16_rne(dg_normal(c->key, base + (uint64_t)j));
  }
}

void dg_host_fill_normal_rows(uint16_t* out, const int64_t* row_ids, int64_t n_rows, int64_t row_len,
                              uint64_t seed, uint32_t tensor_id, int n_threads) {
  dg_rows_ctx c = {out, dg_stream_key(seed, tensor_id), row_ids, row_len};
  dg_parallel(n_rows, n_threads, dg_rows_body, &c);
}

/* ---- index-query rows with planted needles ------------------------------- */
typedef struct {
  uint16_t* out;
  const int64_t* row_ids;
  const int64_t* pos;
  uint64_t noise_key, pick_key;
  int G, d_I, Bk, m, cap;
  const int32_t* needle_block;
  const float* u;
  float beta;
} dg_qidx_ctx;

static void dg_qidx_body(int64_t lo, int64_t hi, void* p) {
  dg_qidx_ctx* c = (dg_qidx_ctx*)p;
  for (int64_t i = lo; i < hi; ++i) {
    int64_t rr = i / c->G;
    int g = (int)(i % c->G);
    dg_q_idx_row(c->out + i * c->d_I, c->noise_key, c->pick_key, c->row_ids[rr], c->pos[rr], g, c->G,
                 c->d_I, c->Bk, c->m, c->cap, c->needle_block, c->u, c->beta);
  }
}

/*
 * out[rr, g, :] for rr < n_rows: the index-query row of tensor row row_ids[rr]
 * (whose query position is pos[rr]) and group g.
 */
void dg_host_q_idx_rows(uint16_t* out, const int64_t* row_ids, const int64_t* pos, int64_t n_rows,
                        uint64_t seed, uint32_t noise_tid, uint32_t pick_tid, int G, int d_I, int Bk,
                        int m, int cap, const int32_t* needle_block, const float* u, float beta,
                        int n_threads) {
  dg_qidx_ctx c = {out, row_ids, pos, dg_stream_key(seed, noise_tid), dg_stream_key(seed, pick_tid),
                   G, d_I, Bk, m, cap, needle_block, u, beta};
  dg_parallel(n_rows * G, n_threads, dg_qidx_body, &c);
}

/* ---- which needles each index-query row picked (bit n of out[rr*G + g]) -- */
void dg_host_pick_masks(uint32_t* out, const int64_t* row_ids, const int64_t* pos, int64_t n_rows,
                        uint64_t seed, uint32_t pick_tid, int G, int Bk, int m, int cap,
                        const int32_t* needle_block) {
  uint64_t key = dg_stream_key(seed, pick_tid);
  for (int64_t rr = 0; rr < n_rows; ++rr)
    for (int g = 0; g < G; ++g)
      out[rr * G + g] = dg_pick_mask(key, row_ids[rr], pos[rr], g, G, Bk, m, cap, needle_block);
}
