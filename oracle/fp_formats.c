/*
 * fp_formats.c -- oracle encoders and decoders for FP16, BF16, E4M3, E5M2.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Every format is described by its fields, as the pages describe them:
 *   - FP16: 1 sign, 5 exponent, 10 mantissa bits, bias 15; max 65504, min
 *     normal 2^-14, min subnormal 2^-24 ([P3] paragraph quoting NVIDIA's
 *     FP16 bounds; [P5] "Range and precision" self-test answer 1).
 *   - BF16: 1 / 8 / 7 bits, bias 127, FP32's exponent range ([P5] "Range and
 *     precision"; [P1] "The triangle").
 *   - E4M3: 1 / 4 / 3 bits, bias 7, max 448, no infinities, one NaN mantissa
 *     pattern; E5M2: 1 / 5 / 2 bits, bias 15, max 57344, IEEE-style Inf/NaN
 *     ([P3] paragraph on the FP8 specification; [P4] "Failure 2").
 *
 * Decoding is exact (double holds every value of all four formats).
 * Encoding takes the definition literally: find the binade of |v|, count
 * how many quanta of that binade (or of the subnormal range) |v| spans,
 * round that count to the nearest integer with ties to the even count, and
 * rebuild the fields.  All steps are exact in double because every input
 * is an FP32 value.
 */
#include <math.h>
#include <stdint.h>

#include "oracle.h"

typedef struct {
  int ebits;          /* exponent field width                               */
  int mbits;          /* mantissa (trailing significand) field width        */
  int bias;
  int ieee_specials;  /* 1: all-ones exponent holds Inf (m == 0) and NaN    */
                      /* 0: all-ones exponent is a normal binade except the */
                      /*    all-ones mantissa, which is the only NaN (E4M3) */
} fmt_desc;

static const fmt_desc FMT_F16 = {5, 10, 15, 1};
static const fmt_desc FMT_BF16 = {8, 7, 127, 1};
static const fmt_desc FMT_E4M3 = {4, 3, 7, 0};
static const fmt_desc FMT_E5M2 = {5, 2, 15, 1};

static const fmt_desc* fp8_desc(int fmt) { return fmt == ORC_E5M2 ? &FMT_E5M2 : &FMT_E4M3; }

/* Largest finite code of a format, as a field pattern without the sign. */
static uint32_t max_code(const fmt_desc* f) {
  uint32_t emask = (1u << f->ebits) - 1, mmask = (1u << f->mbits) - 1;
  if (f->ieee_specials) return ((emask - 1) << f->mbits) | mmask;  /* S.11110.11 */
  return (emask << f->mbits) | (mmask - 1);                        /* S.1111.110 */
}

static double decode_fields(uint32_t bits, const fmt_desc* f) {
  uint32_t emask = (1u << f->ebits) - 1, mmask = (1u << f->mbits) - 1;
  uint32_t m = bits & mmask;
  uint32_t e = (bits >> f->mbits) & emask;
  uint32_t s = (bits >> (f->mbits + f->ebits)) & 1u;
  double sign = s ? -1.0 : 1.0;
  if (e == emask) {
    if (f->ieee_specials) return m == 0 ? sign * INFINITY : NAN;
    if (m == mmask) return NAN;
  }
  if (e == 0) /* subnormal: m quanta of 2^(1 - bias - mbits) */
    return sign * ldexp((double)m, 1 - f->bias - f->mbits);
  return sign * ldexp((double)(m | (1u << f->mbits)), (int)e - f->bias - f->mbits);
}

static double max_finite(const fmt_desc* f) { return decode_fields(max_code(f), f); }

/* Nearest representable value of format f to v (finite, non-zero magnitude
 * a), ties to the even quantum count; returns the field pattern without the
 * sign, or -1 when the rounded magnitude exceeds the largest finite value. */
static int64_t round_to_fields(double a, const fmt_desc* f) {
  int emin = 1 - f->bias;
  int e;
  frexp(a, &e);
  e -= 1;                                   /* a is in [2^e, 2^(e+1))          */
  if (e < emin) e = emin;                   /* subnormal range: fixed quantum  */
  double quantum = ldexp(1.0, e - f->mbits);
  double n = a / quantum;                   /* exact: divide by a power of two */
  double lo = floor(n);
  double frac = n - lo;
  double k = lo;
  if (frac > 0.5 || (frac == 0.5 && fmod(lo, 2.0) != 0.0)) k = lo + 1.0;
  double r = k * quantum;                   /* the rounded magnitude           */
  if (r > max_finite(f)) return -1;
  if (r < ldexp(1.0, emin))                 /* subnormal (or zero) result      */
    return (int64_t)(r / ldexp(1.0, emin - f->mbits));
  int er;
  frexp(r, &er);
  er -= 1;
  int64_t m = (int64_t)(r / ldexp(1.0, er - f->mbits)) - ((int64_t)1 << f->mbits);
  return ((int64_t)(er + f->bias) << f->mbits) | m;
}

/* IEEE-style encode (FP16, BF16): overflow rounds to Inf, NaN stays NaN. */
static uint32_t encode_ieee(float v, const fmt_desc* f, uint32_t quiet_nan) {
  uint32_t sbit = signbit(v) ? 1u << (f->ebits + f->mbits) : 0u;
  uint32_t inf = ((1u << f->ebits) - 1) << f->mbits;
  if (isnan(v)) return sbit | quiet_nan;
  double a = fabs((double)v);
  if (isinf(a)) return sbit | inf;
  if (a == 0.0) return sbit;
  int64_t fields = round_to_fields(a, f);
  return fields < 0 ? (sbit | inf) : (sbit | (uint32_t)fields);
}

double orc_f16_decode(uint16_t h) { return decode_fields(h, &FMT_F16); }
double orc_bf16_decode(uint16_t b) { return decode_fields(b, &FMT_BF16); }
double orc_fp8_decode(uint8_t c, int fmt) { return decode_fields(c, fp8_desc(fmt)); }
double orc_fp8_max(int fmt) { return max_finite(fp8_desc(fmt)); }

uint16_t orc_f16_encode(float f) { return (uint16_t)encode_ieee(f, &FMT_F16, 0x7E00u); }
uint16_t orc_bf16_encode(float f) { return (uint16_t)encode_ieee(f, &FMT_BF16, 0x7FC0u); }

/* FP8 encode, saturating: any magnitude that rounds beyond the largest
 * finite value (and +-Inf) becomes +-max; every NaN becomes 0x7F. */
uint8_t orc_fp8_encode(float v, int fmt) {
  const fmt_desc* f = fp8_desc(fmt);
  uint32_t sbit = signbit(v) ? 0x80u : 0u;
  if (isnan(v)) return 0x7F;
  double a = fabs((double)v);
  if (isinf(a)) return (uint8_t)(sbit | max_code(f));
  if (a == 0.0) return (uint8_t)sbit;
  int64_t fields = round_to_fields(a, f);
  if (fields < 0) return (uint8_t)(sbit | max_code(f));
  return (uint8_t)(sbit | (uint32_t)fields);
}

/* ---- array helpers -------------------------------------------------- */
static double load_elem(const void* x, int dtype, int64_t i) {
  if (dtype == ORC_F16) return orc_f16_decode(((const uint16_t*)x)[i]);
  if (dtype == ORC_BF16) return orc_bf16_decode(((const uint16_t*)x)[i]);
  return (double)((const float*)x)[i];
}

void orc_decode_array(const void* in, int dtype, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (float)load_elem(in, dtype, i);
}

void orc_encode_array(const float* in, int64_t n, int dtype, void* out) {
  for (int64_t i = 0; i < n; ++i) {
    if (dtype == ORC_F16) ((uint16_t*)out)[i] = orc_f16_encode(in[i]);
    else if (dtype == ORC_BF16) ((uint16_t*)out)[i] = orc_bf16_encode(in[i]);
    else ((float*)out)[i] = in[i];
  }
}

void orc_fp8_encode_array(const float* in, int64_t n, int fmt, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_fp8_encode(in[i], fmt);
}

void orc_fp8_decode_array(const uint8_t* in, int64_t n, int fmt, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (float)orc_fp8_decode(in[i], fmt);
}

/* Exposed for fp8_quant.c. */
double orc__load_elem(const void* x, int dtype, int64_t i) { return load_elem(x, dtype, i); }
