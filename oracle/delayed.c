/*
 * delayed.c -- oracle for the two policies named beside the main path.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * 1. Delayed per-tensor scaling ([P4] "Why FP8 training is stable",
 *    "Failure 1": keep a short history of recent max-abs values and derive
 *    s from it, so the scale applied this step comes from what the tensor
 *    looked like on earlier steps; [P5] "FP8 training" figure: per tensor,
 *    delayed, from recent amax).  Readings taken:
 *      s_k = max(max(history), 1e-12) / MAX  (fp32; the history's max is
 *            NaN-propagating like every amax here),
 *      q   = fp8(clamp(x / s_k))             (RNE, saturating),
 *      then this step's amax is written at history[pos], pos = (pos+1) % H.
 *    A zero history gives the floor scale, so the first step saturates
 *    every non-tiny value: the pages' warning taken literally.
 *
 * 2. A loss-scale policy with hysteresis ([P3] "Numerical Precision, Mixed
 *    Precision, and Loss Scaling", DeepSpeed paragraph: loss_scale_window
 *    1000, hysteresis 2, consecutive_hysteresis false, min_loss_scale 1).
 *    The pages give the parameter names only; the reading taken:
 *      overflow:  the step is skipped; the window restarts (tracker = 0);
 *                 if the remaining hysteresis h > 1 it is decremented and S
 *                 kept, otherwise S = max(S * backoff, min_scale);
 *      clean:     tracker += 1; with consecutive_hysteresis h is restored
 *                 to `hysteresis` after every clean step; when tracker
 *                 reaches the window, S *= growth, tracker = 0, and (without
 *                 consecutive_hysteresis) h is restored.
 *    With hysteresis 1 and min_scale 0 this is exactly orc_scaler_update.
 */
#include <math.h>
#include <stdint.h>

#include "oracle.h"

double orc__load_elem(const void* x, int dtype, int64_t i);

void orc_quant_tensor_delayed(const void* x, int dtype, int64_t n, int fmt, float* history,
                              int32_t hist_len, int32_t* pos, uint8_t* q, float* scale_used) {
  float hmax = 0.0f;
  int hnan = 0;
  for (int32_t j = 0; j < hist_len; ++j) {
    if (isnan(history[j])) hnan = 1;
    else if (history[j] > hmax) hmax = history[j];
  }
  float s = orc_scale_from_amax(hnan ? NAN : hmax, fmt);
  *scale_used = s;
  for (int64_t i = 0; i < n; ++i) q[i] = orc_quant_one((float)orc__load_elem(x, dtype, i), s, fmt);
  history[*pos] = orc_amax(x, dtype, n);
  *pos = (*pos + 1) % hist_len;
}

void orc_scaler_update_hysteresis(float* scale, int32_t* tracker, int32_t* hyst, int64_t* skipped,
                                  int32_t found, float growth_factor, float backoff_factor,
                                  int32_t window, int32_t hysteresis, int32_t consecutive,
                                  float min_scale) {
  if (found) {
    if (skipped) *skipped += 1;
    *tracker = 0;
    if (*hyst > 1) {
      *hyst -= 1;
    } else {
      float s = *scale * backoff_factor;
      *scale = s < min_scale ? min_scale : s;
    }
    return;
  }
  *tracker += 1;
  if (consecutive) *hyst = hysteresis;
  if (*tracker >= window) {
    *scale = *scale * growth_factor;
    *tracker = 0;
    if (!consecutive) *hyst = hysteresis;
  }
}
