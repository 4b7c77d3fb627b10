/*
 * mx_quant.c -- oracle for MXFP8: FP8 elements sharing one power-of-two
 * scale per 32 consecutive elements.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * [P5] "Mixed precision and FP8 training", section "FP8 training", notes
 * that Blackwell's MX formats keep one scaling factor per 32 elements in
 * hardware.  The pages give no more than that; the rest of this file is the
 * plainest reading consistent with it (the OCP Microscaling convention),
 * and its parity with the pages is therefore unpinned beyond the block
 * size:
 *   - the scale is a power of two X = 2^e stored as an 8-bit exponent with
 *     bias 127 (E8M0: code c means 2^(c-127), code 255 is NaN);
 *   - e = floor(log2(amax)) - emax_elem, with emax_elem the exponent of the
 *     element format's largest binade (8 for E4M3, 15 for E5M2), clamped to
 *     [-127, 127]; an all-zero block takes e = -127;
 *   - every element is cast as fp8(V / X), round to nearest even,
 *     saturating at +-MAX (V / X can reach just under 2^(emax_elem+1));
 *   - a block holding Inf or NaN gets the NaN scale 255 and all its codes
 *     are 0x7F;
 *   - dequantise: y = decode(q) * 2^e in fp32 (bf16 optionally, RNE).
 */
#include <math.h>
#include <stdint.h>

#include "oracle.h"

double orc__load_elem(const void* x, int dtype, int64_t i);

double orc_e8m0_decode(uint8_t c) {
  if (c == 255) return NAN;
  return ldexp(1.0, (int)c - 127);
}

static int emax_elem(int fmt) { return fmt == ORC_E5M2 ? 15 : 8; }

/* E8M0 code of the shared scale of a block with this amax (-1 = NaN). */
int32_t orc_mx_scale_code(double amax, int fmt) {
  if (isnan(amax) || isinf(amax)) return 255;
  int e;
  if (amax == 0.0) {
    e = -127;
  } else {
    int k;
    frexp(amax, &k);       /* amax = m * 2^k, m in [0.5, 1) */
    e = (k - 1) - emax_elem(fmt);
    if (e < -127) e = -127;
    if (e > 127) e = 127;
  }
  return e + 127;
}

void orc_quant_mx(const void* x, int dtype, int64_t R, int64_t C, int fmt, uint8_t* q,
                  uint8_t* scales) {
  const int64_t nb = C / 32;
  for (int64_t r = 0; r < R; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      const int64_t base = r * C + b * 32;
      double amax = 0.0;
      int special = 0;
      for (int64_t i = 0; i < 32; ++i) {
        double v = fabs(orc__load_elem(x, dtype, base + i));
        if (isnan(v) || isinf(v)) special = 1;
        else if (v > amax) amax = v;
      }
      int32_t code = special ? 255 : orc_mx_scale_code(amax, fmt);
      scales[r * nb + b] = (uint8_t)code;
      for (int64_t i = 0; i < 32; ++i) {
        if (code == 255) {
          q[base + i] = 0x7F;
          continue;
        }
        /* V / X with X a power of two: exact in double, one rounding to fp32 */
        float v = (float)ldexp(orc__load_elem(x, dtype, base + i), 127 - code);
        q[base + i] = orc_fp8_encode(v, fmt);   /* RNE, saturating */
      }
    }
}

void orc_dequant_mx(const uint8_t* q, const uint8_t* scales, int64_t R, int64_t C, int fmt,
                    int out_dtype, void* y) {
  const int64_t nb = C / 32;
  for (int64_t r = 0; r < R; ++r)
    for (int64_t c = 0; c < C; ++c) {
      float s = (float)orc_e8m0_decode(scales[r * nb + c / 32]);
      float v = (float)orc_fp8_decode(q[r * C + c], fmt) * s;
      if (out_dtype == ORC_BF16) ((uint16_t*)y)[r * C + c] = orc_bf16_encode(v);
      else ((float*)y)[r * C + c] = v;
    }
}
