/*
 * fp8_quant.c -- oracle for FP8 quantisation with fine-grained scaling.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Restates [P5] "FP8 training", the fp8_scaling.py listing:
 *   quant(x, s)      = clamp(x / s, -MAX, MAX) cast to FP8; dequantised as
 *                      decode(q) * s;
 *   per_block(x,r,c) = reshape [R, C] into (R/r, r, C/c, c), take max |x|
 *                      over each r x c block, clamp it below at 1e-12,
 *                      divide by MAX: that is the block's FP32 scale;
 *   per_tensor(x)    = the same with a single block covering the tensor.
 * The tile shapes are [P1]/[P4]/[P5]'s: 1 x 128 for activations (one row,
 * 128 consecutive channels) and 128 x 128 for weights; [P4] "Failure 1"
 * gives the current-scaling rule (scale from this tensor's own amax,
 * multiply by s on the way out).
 *
 * Readings (the pages leave these open):
 *   - The per-tensor scale gets the same 1e-12 floor as the block scale, so
 *     an all-zero tensor quantises to zeros instead of NaN.
 *   - A NaN anywhere in a block makes amax NaN (max propagates NaN), hence
 *     s NaN and every code of that block 0x7F.  An Inf makes s = +Inf, so
 *     finite elements give +-0 and the Inf itself Inf/Inf = NaN -> 0x7F.
 *   - All FP8 NaNs are written as 0x7F (sign dropped).
 *   - Dequantise computes decode(q) * s in fp32; the bfloat16 output form
 *     rounds that fp32 product to nearest even.
 */
#include <math.h>
#include <stdint.h>

#include "oracle.h"

double orc__load_elem(const void* x, int dtype, int64_t i);

static float block_amax(const void* x, int dtype, int64_t C, int64_t r0, int64_t c0,
                        int64_t br, int64_t bc) {
  float amax = 0.0f;
  for (int64_t r = r0; r < r0 + br; ++r)
    for (int64_t c = c0; c < c0 + bc; ++c) {
      double v = fabs(orc__load_elem(x, dtype, r * C + c));
      if (isnan(v)) return NAN;
      if (v > amax) amax = (float)v;
    }
  return amax;
}

float orc_amax(const void* x, int dtype, int64_t n) {
  return n == 0 ? 0.0f : block_amax(x, dtype, n, 0, 0, 1, n);
}

float orc_scale_from_amax(float amax, int fmt) {
  const float floor_amax = 1e-12f;
  float a = amax;
  if (!isnan(a) && a < floor_amax) a = floor_amax;
  return a / (float)orc_fp8_max(fmt);
}

uint8_t orc_quant_one(float x, float s, int fmt) {
  const float mx = (float)orc_fp8_max(fmt);
  float v = x / s;
  if (v > mx) v = mx;
  if (v < -mx) v = -mx;
  return orc_fp8_encode(v, fmt);
}

void orc_quant_block(const void* x, int dtype, int64_t R, int64_t C, int64_t br,
                     int64_t bc, int fmt, uint8_t* q, float* scales) {
  int64_t nbc = C / bc;
  for (int64_t bi = 0; bi < R / br; ++bi)
    for (int64_t bj = 0; bj < nbc; ++bj) {
      float s = orc_scale_from_amax(block_amax(x, dtype, C, bi * br, bj * bc, br, bc), fmt);
      scales[bi * nbc + bj] = s;
      for (int64_t r = bi * br; r < (bi + 1) * br; ++r)
        for (int64_t c = bj * bc; c < (bj + 1) * bc; ++c)
          q[r * C + c] = orc_quant_one((float)orc__load_elem(x, dtype, r * C + c), s, fmt);
    }
}

void orc_quant_tensor(const void* x, int dtype, int64_t n, int fmt, uint8_t* q,
                      float* scale) {
  float s = orc_scale_from_amax(orc_amax(x, dtype, n), fmt);
  *scale = s;
  for (int64_t i = 0; i < n; ++i) q[i] = orc_quant_one((float)orc__load_elem(x, dtype, i), s, fmt);
}

void orc_dequant(const uint8_t* q, const float* scales, int64_t R, int64_t C, int64_t br,
                 int64_t bc, int fmt, int out_dtype, void* y) {
  int64_t nbc = C / bc;
  for (int64_t r = 0; r < R; ++r)
    for (int64_t c = 0; c < C; ++c) {
      float s = scales[(r / br) * nbc + c / bc];
      float v = (float)orc_fp8_decode(q[r * C + c], fmt) * s;
      if (out_dtype == ORC_BF16) ((uint16_t*)y)[r * C + c] = orc_bf16_encode(v);
      else ((float*)y)[r * C + c] = v;
    }
}
