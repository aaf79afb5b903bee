/*
 * Seeded synthetic-input generator: the arithmetic shared by the host (C) and
 * device (CUDA) fill routines, so that both produce bit-identical tensors.
 *
 * This file holds no part of the sparse-attention method: only a
 * counter-based random source and the rounding to bf16.
 *
 *   mix64      : the SplitMix64 finaliser (Steele, Lea, Flood, "Fast
 *                splittable pseudorandom number generators", OOPSLA 2014).
 *   word(i, w) : mix64(key + (2i + w) * golden_gamma), key = per-tensor stream.
 *   normal(i)  : Irwin-Hall sum of the eight 16-bit lanes of word(i,0) and
 *                word(i,1), centred and scaled to unit variance in fp32
 *                (integer arithmetic until one exact int->fp32 conversion and
 *                one correctly rounded fp32 multiply).  Approximately N(0,1),
 *                bounded by +-4.9.
 *   bit(i)     : the top bit of word(i, 0).
 *   bf16_rne   : fp32 -> bf16, round to nearest even (inputs are never NaN).
 *
 * Every step is integer or a single IEEE-rounded fp32 operation, so the host
 * and device versions agree bit for bit.
 */
#ifndef MSA_DATAGEN_CORE_H
#define MSA_DATAGEN_CORE_H

#include <stdint.h>

#if defined(__CUDACC__)
#define DG_FN __host__ __device__ __forceinline__
#else
#define DG_FN static inline
#endif

#define DG_GAMMA 0x9E3779B97F4A7C15ULL
#define DG_IH_MEAN 262140          /* 8 * 65535 / 2 */
#define DG_IH_SCALE_BITS 0x379cc471u /* fp32(1 / sqrt(8 * (65536^2 - 1) / 12)) */

DG_FN uint64_t dg_mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

DG_FN uint64_t dg_stream_key(uint64_t seed, uint32_t tensor_id) {
  return dg_mix64(seed * DG_GAMMA + (uint64_t)tensor_id * 0xD1B54A32D192ED03ULL +
                  0x5851F42D4C957F2DULL);
}

DG_FN uint64_t dg_word(uint64_t key, uint64_t i, uint32_t w) {
  return dg_mix64(key + (2ULL * i + (uint64_t)w) * DG_GAMMA);
}

DG_FN int32_t dg_lane_sum(uint64_t z) {
  return (int32_t)((z & 0xFFFFu) + ((z >> 16) & 0xFFFFu) + ((z >> 32) & 0xFFFFu) +
                   ((z >> 48) & 0xFFFFu));
}

DG_FN float dg_bits_to_float(uint32_t b) {
#if defined(__CUDA_ARCH__)
  return __uint_as_float(b);
#else
  union { uint32_t u; float f; } c;
  c.u = b;
  return c.f;
#endif
}

DG_FN uint32_t dg_float_to_bits(float f) {
#if defined(__CUDA_ARCH__)
  return __float_as_uint(f);
#else
  union { uint32_t u; float f; } c;
  c.f = f;
  return c.u;
#endif
}

/* fp32 multiply / add with one rounding each (no contraction into an FMA). */
DG_FN float dg_mul(float a, float b) {
#if defined(__CUDA_ARCH__)
  return __fmul_rn(a, b);
#else
  volatile float r = a * b;
  return r;
#endif
}

DG_FN float dg_add(float a, float b) {
#if defined(__CUDA_ARCH__)
  return __fadd_rn(a, b);
#else
  volatile float r = a + b;
  return r;
#endif
}

DG_FN float dg_normal(uint64_t key, uint64_t i) {
  int32_t s = dg_lane_sum(dg_word(key, i, 0)) + dg_lane_sum(dg_word(key, i, 1)) - DG_IH_MEAN;
  /* |s| <= 262140 < 2^24: the conversion is exact. */
  return dg_mul((float)s, dg_bits_to_float(DG_IH_SCALE_BITS));
}

DG_FN uint32_t dg_bit(uint64_t key, uint64_t i) {
  return (uint32_t)(dg_word(key, i, 0) >> 63);
}

DG_FN uint16_t dg_bf16_rne(float f) {
  uint32_t b = dg_float_to_bits(f);
  b += 0x7FFFu + ((b >> 16) & 1u);
  return (uint16_t)(b >> 16);
}

/*
 * Index-query row with planted needles.  For row r (position t) and group g:
 *   C = the first `cap` needles n (in increasing n) of group g whose block lies
 *       strictly before local(t) = t / Bk and whose pick bit is set,
 *   usum = sum over n in C of u[g*m + n] (fp32, increasing n),
 *   q_idx = bf16(x + beta * usum)   (x = the row's normal noise),
 * or bf16(x) when C is empty.  Writes d_I bf16 values to out.
 */
DG_FN uint32_t dg_pick_mask(uint64_t pick_key, int64_t r, int64_t t, int g, int G, int Bk, int m,
                            int cap, const int32_t* needle_block /*[G*m]*/) {
  int64_t local = t / Bk;
  uint32_t picked = 0; /* bit n set if needle n is in C (m <= 32) */
  int n_picked = 0;
  for (int n = 0; n < m && n_picked < cap; ++n) {
    if ((int64_t)needle_block[g * m + n] >= 0 && (int64_t)needle_block[g * m + n] < local &&
        dg_bit(pick_key, ((uint64_t)r * (uint64_t)G + (uint64_t)g) * (uint64_t)m + (uint64_t)n)) {
      picked |= 1u << n;
      ++n_picked;
    }
  }
  return picked;
}

DG_FN void dg_q_idx_row(uint16_t* out, uint64_t noise_key, uint64_t pick_key, int64_t r,
                        int64_t t, int g, int G, int d_I, int Bk, int m, int cap,
                        const int32_t* needle_block /*[G*m]*/, const float* u /*[G*m, d_I]*/,
                        float beta) {
  uint64_t base = ((uint64_t)r * (uint64_t)G + (uint64_t)g) * (uint64_t)d_I;
  uint32_t picked = dg_pick_mask(pick_key, r, t, g, G, Bk, m, cap, needle_block);
  for (int c = 0; c < d_I; ++c) {
    float x = dg_normal(noise_key, base + (uint64_t)c);
    if (picked) {
      float us = 0.0f;
      for (int n = 0; n < m; ++n)
        if (picked & (1u << n)) us = dg_add(us, u[(int64_t)(g * m + n) * d_I + c]);
      x = dg_add(x, dg_mul(beta, us));
    }
    out[c] = dg_bf16_rne(x);
  }
}

#endif /* MSA_DATAGEN_CORE_H */
