/*
 * master.c -- oracle for the consumer of the unscaled gradients: the
 * global gradient norm, clipping and the FP32 master-weight update that is
 * skipped on overflow.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * [P3] "Numerical Precision, Mixed Precision, and Loss Scaling", the
 * six-step training step, step 5: clip and update -- apply guardrails,
 * write into FP32 master state, and skip invalid steps; and the paragraph on
 * skipped updates (whatever consumes the step must agree on whether a real
 * optimizer step occurred).  [P5] "Mixed precision and FP8 training",
 * "Range and precision": the optimizer updates FP32 master weights and
 * converts them to bf16 each step for the forward pass.  [P2] "Where it
 * fits": loss scaling pairs with gradient clipping.
 * Readings taken:
 *   norm  = sqrt(sum of g_i^2) over every unscaled gradient (the plain
 *           definition, computed here with compensated double sums);
 *   coef  = max_norm / norm when max_norm > 0 and norm > max_norm, else 1
 *           (fp32 division);
 *   SGD:  w = w - lr * (coef * g), each product and the difference rounded
 *         to fp32 separately (no fused multiply-add); the bf16 copy is w
 *         rounded to nearest even;
 *   a step with found_inf set changes nothing.
 */
#include <math.h>
#include <stdint.h>

#include "oracle.h"

double orc_sum_squares(const float* g, int64_t n) {
  double sum = 0.0, c = 0.0;  /* Neumaier compensated summation */
  for (int64_t i = 0; i < n; ++i) {
    double v = (double)g[i] * (double)g[i];   /* exact: 24-bit x 24-bit < 53 bits */
    double t = sum + v;
    if (fabs(sum) >= fabs(v)) c += (sum - t) + v;
    else c += (v - t) + sum;
    sum = t;
  }
  return sum + c;
}

float orc_clip_coef(float norm, float max_norm) {
  if (max_norm > 0.0f && norm > max_norm) return max_norm / norm;
  return 1.0f;
}

void orc_master_update_sgd(float* w, uint16_t* w_bf16, const float* g, int64_t n, float lr,
                           float coef, int32_t found_inf) {
  if (found_inf) return;
  for (int64_t i = 0; i < n; ++i) {
    float t1 = coef * g[i];
    float t2 = lr * t1;
    w[i] = w[i] - t2;
    if (w_bf16) w_bf16[i] = orc_bf16_encode(w[i]);
  }
}
