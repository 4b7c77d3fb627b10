/*
 * oracle.h -- plain, slow, scalar CPU oracle for the mixed-precision
 * cast-and-scale path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link
 * or call this code: only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no source, header, table
 * or constant with the CUDA library; the two are compared output by output.
 *
 * Everything here follows the definitions printed on these pages:
 *   [P1] "Loss scaling, FP8, and the failure that never crashes"
 *   [P2] "Loss Scaling" (glossary entry)
 *   [P3] "Numerical Precision, Mixed Precision, and Loss Scaling"
 *   [P4] "Why FP8 training is stable"
 *   [P5] "Mixed precision and FP8 training"
 * Each function below names the section it restates.
 *
 * Arithmetic: fp32 where the pages fix fp32 (the unscale in FP32, the FP32
 * block scale, the FP32 quotient x/s that the FP8 cast consumes); all format
 * decoding is exact via double; all encoders work from the format
 * definitions (sign / exponent / mantissa fields, bias, round to nearest,
 * ties to even) with exact double arithmetic.  Build with
 * -ffp-contract=off so that no multiply-add is fused.
 */
#ifndef GS_ORACLE_H
#define GS_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types of the oracle's array arguments (its own numbering). */
enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_F32 = 2 };
/* The two OCP FP8 encodings. */
enum { ORC_E4M3 = 0, ORC_E5M2 = 1 };

/* ---- number formats ([P3] FP8 specification paragraph; [P3] FP16 bounds
 *      paragraph; [P5] "Range and precision") -------------------------- */
double   orc_f16_decode(uint16_t h);
double   orc_bf16_decode(uint16_t b);
double   orc_fp8_decode(uint8_t c, int fmt);
uint16_t orc_f16_encode(float f);   /* IEEE binary16, RNE, overflow -> Inf   */
uint16_t orc_bf16_encode(float f);  /* bfloat16, RNE, overflow -> Inf         */
uint8_t  orc_fp8_encode(float f, int fmt); /* RNE, saturating, NaN -> 0x7F  */
double   orc_fp8_max(int fmt);      /* 448 or 57344                          */

/* Array helpers (loops over the scalar functions above). */
void orc_decode_array(const void* in, int dtype, int64_t n, float* out);
void orc_encode_array(const float* in, int64_t n, int dtype, void* out);
void orc_fp8_encode_array(const float* in, int64_t n, int fmt, uint8_t* out);
void orc_fp8_decode_array(const uint8_t* in, int64_t n, int fmt, float* out);

/* ---- dynamic loss scaling ([P1] "Loss scaling, derived from the chain
 *      rule you already have" and the SimpleGradScaler listing; [P3]
 *      GradScaler defaults paragraph) -------------------------------------- */

/* out[i] = fp32(g[i]) * fp32(1/S); returns 1 if any g[i] is Inf or NaN. */
int32_t orc_unscale_check(const uint16_t* g, int64_t n, float scale, float* out);
/* S/tracker update after one step; found = OR of the step's flags. */
void orc_scaler_update(float* scale, int32_t* growth_tracker, int64_t* skipped,
                       int32_t found, float growth_factor, float backoff_factor,
                       int32_t growth_interval);
/* One whole step over a list of tensors: unscale every tensor, OR the flags,
 * update the state.  Returns the step's found flag. */
int32_t orc_gradscaler_step(const uint16_t* const* g, float* const* out,
                            const int64_t* numel, int32_t n_tensors,
                            float* scale, int32_t* growth_tracker, int64_t* skipped,
                            float growth_factor, float backoff_factor,
                            int32_t growth_interval);

/* ---- FP8 quantisation with fine-grained scaling ([P5] "FP8 training",
 *      the fp8_scaling.py listing's quant / per_tensor / per_block; [P4]
 *      "Failure 1" and "The seam"; [P1] "FP8 needs a finer-grained fix") -- */

/* Block amax, FP32 block scale and FP8 codes for a row-major [R, C] array
 * cut into br x bc blocks (br | R, bc | C).  scales is [R/br, C/bc]. */
void orc_quant_block(const void* x, int dtype, int64_t R, int64_t C,
                     int64_t br, int64_t bc, int fmt, uint8_t* q, float* scales);
/* One scale for the whole tensor of n elements. */
void orc_quant_tensor(const void* x, int dtype, int64_t n, int fmt,
                      uint8_t* q, float* scale);
/* y = decode(q) * s (fp32), then optionally bfloat16 (out_dtype ORC_BF16). */
void orc_dequant(const uint8_t* q, const float* scales, int64_t R, int64_t C,
                 int64_t br, int64_t bc, int fmt, int out_dtype, void* y);

/* ---- MXFP8: one power-of-two (E8M0) scale per 32 consecutive elements
 *      ([P5] "FP8 training", the MX formats sentence; see mx_quant.c) ---- */
double  orc_e8m0_decode(uint8_t c);
int32_t orc_mx_scale_code(double amax, int fmt);
void orc_quant_mx(const void* x, int dtype, int64_t R, int64_t C, int fmt, uint8_t* q,
                  uint8_t* scales);
void orc_dequant_mx(const uint8_t* q, const uint8_t* scales, int64_t R, int64_t C, int fmt,
                    int out_dtype, void* y);

/* ---- delayed per-tensor scaling and a hysteresis loss-scale policy
 *      ([P4] "Failure 1"; [P3] DeepSpeed paragraph; see delayed.c) ------- */
void orc_quant_tensor_delayed(const void* x, int dtype, int64_t n, int fmt, float* history,
                              int32_t hist_len, int32_t* pos, uint8_t* q, float* scale_used);
void orc_scaler_update_hysteresis(float* scale, int32_t* tracker, int32_t* hyst, int64_t* skipped,
                                  int32_t found, float growth_factor, float backoff_factor,
                                  int32_t window, int32_t hysteresis, int32_t consecutive,
                                  float min_scale);

/* ---- the consumer step: global gradient norm, clipping, FP32 master
 *      weights ([P3] six-step training step, step 5; [P5] "Range and
 *      precision"; see master.c) ------------------------------------------ */
double orc_sum_squares(const float* g, int64_t n);
float  orc_clip_coef(float norm, float max_norm);
void   orc_master_update_sgd(float* w, uint16_t* w_bf16, const float* g, int64_t n, float lr,
                             float coef, int32_t found_inf);

/* ---- the GEMM that consumes the tiles, FP32 promotion every 128 of K
 *      ([P1] "FP8 needs a finer-grained fix"; [P5] "FP8 training"; see
 *      gemm.c) ------------------------------------------------------------ */
double orc_gemm_fp8_block_elem(const uint8_t* qa, const float* sa, const uint8_t* qb,
                               const float* sb, int64_t K, int64_t m, int64_t n, int fmt_a,
                               int fmt_b);
void orc_gemm_fp8_block(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                        int64_t M, int64_t N, int64_t K, int fmt_a, int fmt_b, double* d);

/* Pieces of the block path, exposed so tests can pin each step. */
float orc_amax(const void* x, int dtype, int64_t n);          /* NaN-propagating */
float orc_scale_from_amax(float amax, int fmt);               /* max(a,1e-12)/MAX */
uint8_t orc_quant_one(float x, float s, int fmt);              /* enc(clamp(x/s))  */

#ifdef __cplusplus
}
#endif
#endif
