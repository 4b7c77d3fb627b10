/*
 * gradscaler.c -- oracle for the dynamic loss scaler's per-step bookkeeping.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * Restates:
 *   [P1] "Loss scaling, derived from the chain rule you already have":
 *        gradients come out of backward multiplied by S; each one is divided
 *        by S again, in FP32, before the optimizer; if any gradient is Inf
 *        or NaN the step is skipped and S is halved; after enough clean steps
 *        S is multiplied by the growth factor.
 *   [P1] SimpleGradScaler listing: the overflow test runs on the scaled
 *        gradients before unscaling; a clean step increments the clean-step
 *        counter, and when the counter reaches growth_interval S grows and
 *        the counter returns to 0; an overflow resets the counter to 0.
 *   [P3] GradScaler defaults paragraph: init 65536, growth 2.0, backoff 0.5,
 *        growth_interval 2000 (the backoff factor replaces the listing's
 *        hard-coded division by 2).
 *
 * Readings (the pages leave these open):
 *   - "divide by S in FP32" is computed as fp32(g) * fp32(1/S) with the
 *     reciprocal formed in double and rounded once to fp32.  For a power-of-
 *     two S (every S this loop can reach from a power-of-two start with
 *     factors 2 and 0.5) this equals the fp32 division exactly.
 *   - The unscaled output is written on skipped steps too; the caller skips
 *     the optimizer.
 *   - Growth is applied as written, with no guard against S overflowing.
 */
#include <math.h>
#include <stdint.h>

#include "oracle.h"

int32_t orc_unscale_check(const uint16_t* g, int64_t n, float scale, float* out) {
  float inv_scale = (float)(1.0 / (double)scale);
  int32_t found = 0;
  for (int64_t i = 0; i < n; ++i) {
    double v = orc_f16_decode(g[i]);
    if (isinf(v) || isnan(v)) found = 1;
    out[i] = (float)v * inv_scale;
  }
  return found;
}

void orc_scaler_update(float* scale, int32_t* growth_tracker, int64_t* skipped,
                       int32_t found, float growth_factor, float backoff_factor,
                       int32_t growth_interval) {
  if (found) {
    *scale = *scale * backoff_factor;
    *growth_tracker = 0;
    if (skipped) *skipped += 1;
    return;
  }
  *growth_tracker += 1;
  if (*growth_tracker >= growth_interval) {
    *scale = *scale * growth_factor;
    *growth_tracker = 0;
  }
}

int32_t orc_gradscaler_step(const uint16_t* const* g, float* const* out,
                            const int64_t* numel, int32_t n_tensors,
                            float* scale, int32_t* growth_tracker, int64_t* skipped,
                            float growth_factor, float backoff_factor,
                            int32_t growth_interval) {
  int32_t found = 0;
  for (int32_t t = 0; t < n_tensors; ++t)
    if (orc_unscale_check(g[t], numel[t], *scale, out[t])) found = 1;
  orc_scaler_update(scale, growth_tracker, skipped, found, growth_factor, backoff_factor,
                    growth_interval);
  return found;
}
