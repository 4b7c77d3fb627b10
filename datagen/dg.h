/*
 * dg.h -- seeded, counter-based synthetic inputs for the cast-and-scale
 * path.  Shared by the CPU oracle's tests and the GPU benchmarks: this
 * module produces input bit patterns only and holds none of the method's
 * arithmetic (no unscale, no amax, no FP8 rounding, no RNE encoder).
 *
 * Every element is a pure function of (seed, stream, index), so the host
 * and the device produce identical bits and any element of a huge tensor
 * can be regenerated on the host alone.
 *
 * The hash is SplitMix64's finaliser (Steele, Lea and Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014, with Stafford's
 * "Mix13" constants), applied to a counter.
 *
 * Distributions (values are built from integer fields, never by a rounding
 * conversion, so that host and device agree bit for bit):
 *   DG_LOGU_F16 / DG_LOGU_BF16 -- random sign; binade E drawn uniformly
 *       from [e_lo, e_hi]; significand uniform inside the binade (a
 *       log-uniform magnitude at binade resolution).  FP16 binades below
 *       2^-14 are written as the FP16 subnormal pattern of 1.m * 2^E with
 *       the bits below 2^-24 dropped.
 *   DG_NORMAL_BF16 -- Irwin-Hall: the sum of twelve 16-bit uniforms,
 *       centred and divided by 2^16 (an approximately N(0,1) value with
 *       tails cut at +-6), times sigma and times an outlier multiplier, in
 *       fp32; the bfloat16 pattern is the top half of that fp32 word
 *       (truncation, not rounding).
 * Outliers (DG_NORMAL_BF16 only): an element is an outlier with
 * probability elem_p (its value times elem_mult); listed channels (index
 * mod cols) are multiplied by their chan_mult; listed blocks of
 * block_rows x block_cols are multiplied by block_mult.
 */
#ifndef GS_DATAGEN_DG_H
#define GS_DATAGEN_DG_H

#include <stdint.h>
#include <string.h>

#ifdef __CUDACC__
#define DG_HD __host__ __device__ __forceinline__
#else
#define DG_HD static inline
#endif

enum { DG_LOGU_F16 = 0, DG_LOGU_BF16 = 1, DG_NORMAL_BF16 = 2 };

#define DG_MAX_CHAN 16
#define DG_MAX_BLOCKS 64

typedef struct dg_spec {
  uint64_t seed;
  uint64_t stream;             /* tensor id, step id, ... */
  int32_t kind;
  int32_t e_lo, e_hi;          /* binade range of the log-uniform kinds */
  float sigma;                 /* normal kind */
  int64_t cols;                /* row length, for channel / block outliers */
  uint64_t elem_threshold;     /* elem_p * 2^64; 0 = no element outliers */
  float elem_mult;
  int32_t n_chan;
  int64_t chan_id[DG_MAX_CHAN];
  float chan_mult[DG_MAX_CHAN];
  int32_t n_block;
  int32_t block_rows, block_cols;
  float block_mult;
  int64_t block_id[DG_MAX_BLOCKS]; /* (row / block_rows) * (cols / block_cols) + col / block_cols */
} dg_spec;

DG_HD uint64_t dg_mix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* The k-th 64-bit draw of element `index` in stream `stream` of `seed`. */
DG_HD uint64_t dg_draw(uint64_t seed, uint64_t stream, uint64_t index, uint64_t k) {
  uint64_t key = dg_mix64(seed ^ dg_mix64(stream * 0xD1B54A32D192ED03ull + k));
  return dg_mix64(key + index);
}

DG_HD uint32_t dg_f32_bits(float f) {
#ifdef __CUDA_ARCH__
  return __float_as_uint(f);
#else
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
#endif
}

/* One correctly rounded fp32 product (the host side is compiled with
 * -ffp-contract=off; there is no addition to fuse with anyway). */
DG_HD float dg_mul(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fmul_rn(a, b);
#else
  return a * b;
#endif
}

DG_HD uint16_t dg_logu_f16(const dg_spec* s, uint64_t i) {
  uint64_t h = dg_draw(s->seed, s->stream, i, 0);
  uint32_t sign = (uint32_t)(h >> 63) << 15;
  uint32_t span = (uint32_t)(s->e_hi - s->e_lo + 1);
  int32_t e = s->e_lo + (int32_t)((uint32_t)(h >> 32) % span);
  uint32_t mant = (uint32_t)(h >> 8) & 0x3FFu;
  if (e >= -14) return (uint16_t)(sign | ((uint32_t)(e + 15) << 10) | mant);
  int32_t shift = -14 - e;
  if (shift > 10) return (uint16_t)sign;
  return (uint16_t)(sign | ((0x400u | mant) >> shift));
}

DG_HD uint16_t dg_logu_bf16(const dg_spec* s, uint64_t i) {
  uint64_t h = dg_draw(s->seed, s->stream, i, 0);
  uint32_t sign = (uint32_t)(h >> 63) << 15;
  uint32_t span = (uint32_t)(s->e_hi - s->e_lo + 1);
  int32_t e = s->e_lo + (int32_t)((uint32_t)(h >> 32) % span);
  uint32_t mant = (uint32_t)(h >> 8) & 0x7Fu;
  return (uint16_t)(sign | ((uint32_t)(e + 127) << 7) | mant);
}

DG_HD float dg_outlier_mult(const dg_spec* s, uint64_t i) {
  float m = 1.0f;
  if (s->elem_threshold && dg_draw(s->seed, s->stream, i, 4) < s->elem_threshold) m = s->elem_mult;
  if (s->n_chan > 0) {
    int64_t c = (int64_t)(i % (uint64_t)s->cols);
    for (int k = 0; k < s->n_chan; ++k)
      if (s->chan_id[k] == c) m = dg_mul(m, s->chan_mult[k]);
  }
  if (s->n_block > 0) {
    int64_t r = (int64_t)(i / (uint64_t)s->cols), c = (int64_t)(i % (uint64_t)s->cols);
    int64_t b = (r / s->block_rows) * (s->cols / s->block_cols) + c / s->block_cols;
    for (int k = 0; k < s->n_block; ++k)
      if (s->block_id[k] == b) m = dg_mul(m, s->block_mult);
  }
  return m;
}

DG_HD uint16_t dg_normal_bf16(const dg_spec* s, uint64_t i) {
  int32_t sum = 0;
  for (uint64_t k = 0; k < 3; ++k) {
    uint64_t h = dg_draw(s->seed, s->stream, i, 1 + k);
    sum += (int32_t)(h & 0xFFFF) + (int32_t)((h >> 16) & 0xFFFF) + (int32_t)((h >> 32) & 0xFFFF) +
           (int32_t)(h >> 48);
  }
  int32_t centred = 2 * sum - 12 * 65535;      /* |centred| <= 786420 < 2^24: exact */
  float z = (float)centred * (1.0f / 131072.0f); /* exact: power-of-two scaling */
  float v = dg_mul(dg_mul(z, s->sigma), dg_outlier_mult(s, i));
  return (uint16_t)(dg_f32_bits(v) >> 16);
}

DG_HD uint16_t dg_value(const dg_spec* s, uint64_t i) {
  if (s->kind == DG_LOGU_F16) return dg_logu_f16(s, i);
  if (s->kind == DG_LOGU_BF16) return dg_logu_bf16(s, i);
  return dg_normal_bf16(s, i);
}

#endif
