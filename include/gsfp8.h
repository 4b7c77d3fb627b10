/*
 * gsfp8.h -- C ABI of the GB300 (sm_103a) mixed-precision cast-and-scale
 * library: dynamic loss scaling of FP16 gradient lists and FP8
 * quantisation with fine-grained (1x128 / 128x128 / per-tensor) scaling.
 *
 * Sources of the definitions (web pages, cited by title and section):
 *   [P1] "Loss scaling, FP8, and the failure that never crashes"
 *   [P3] "Numerical Precision, Mixed Precision, and Loss Scaling"
 *   [P4] "Why FP8 training is stable"
 *   [P5] "Mixed precision and FP8 training"
 *
 * Conventions shared by every entry point:
 *   - Return value: a gs_status code.  Argument errors are found on the
 *     host before anything is launched; nothing is enqueued when a call
 *     returns anything but GS_OK.  GS_ERR_CUDA means a CUDA call made by the
 *     library failed (see gs_last_cuda_error).  Nothing throws or aborts.
 *   - Streams: `stream` is a cudaStream_t passed as void*; NULL is the
 *     legacy default stream.  Every compute call is asynchronous on that
 *     stream and never synchronises the host.  The handle is passed to CUDA
 *     as given: it must be a live stream of the current context (CUDA has
 *     no safe check for an arbitrary handle; a launch CUDA refuses returns
 *     GS_ERR_CUDA).
 *   - Memory: every data pointer is device memory of the current device
 *     (or managed memory, or mapped host memory whose device address equals
 *     its host address); pointers the device cannot use as given are
 *     rejected with GS_ERR_ARG.  The caller owns all
 *     data buffers.  The library allocates only inside
 *     gs_tensor_list_create and gs_param_list_create; no compute call
 *     allocates.
 *   - Layout: row-major and contiguous; element [r, c] of an R x C array is
 *     at offset r * C + c.  Outputs must not overlap inputs.  Any element-
 *     aligned address is accepted; 16-byte-aligned buffers take the
 *     vectorised paths.
 *   - Device-side waits are bounded: a kernel that gives up on a wait
 *     records GS_ERR_TIMEOUT in a device status word (gs_device_status)
 *     and returns; it never traps.
 */
#ifndef GSFP8_H
#define GSFP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gs_status {
  GS_OK = 0,
  GS_ERR_NULL = 1,    /* a required pointer is NULL                          */
  GS_ERR_SHAPE = 2,   /* sizes negative, not divisible by the block, too big */
  GS_ERR_DTYPE = 3,   /* unsupported element type or FP8 format              */
  GS_ERR_ARG = 4,     /* other invalid argument (pointer not reachable, ...) */
  GS_ERR_CUDA = 5,    /* a CUDA runtime call failed                          */
  GS_ERR_TIMEOUT = 6  /* a bounded device-side wait expired                  */
} gs_status;

typedef enum gs_dtype { GS_F16 = 0, GS_BF16 = 1, GS_F32 = 2 } gs_dtype;

/* OCP FP8 encodings ([P3] paragraph on the FP8 specification; [P4]
 * "Failure 2"): E4M3 -- bias 7, max 448 (S.1111.110), no infinities, one
 * NaN pattern; E5M2 -- bias 15, max 57344 (S.11110.11), IEEE-style Inf/NaN.
 * Casts are round-to-nearest-even and saturating (|v| beyond max and +-Inf
 * give +-max); every NaN is written as 0x7F. */
typedef enum gs_fp8 { GS_E4M3 = 0, GS_E5M2 = 1 } gs_fp8;

/* Human-readable name of a status code (static string, never NULL). */
const char* gs_status_str(int status);

/* The cudaError_t of the most recent GS_ERR_CUDA on the calling thread. */
int gs_last_cuda_error(void);

/* Library version string. */
const char* gs_version(void);

/* ------------------------------------------------------------------------
 * Dynamic loss scaling ([P1] "Loss scaling, derived from the chain rule you
 * already have" and its SimpleGradScaler listing; [P3] GradScaler defaults
 * paragraph and its six-step training step, step 4 "unscale and inspect"
 * and step 6 "adjust the dynamic loss scale").
 * --------------------------------------------------------------------- */

/* Opaque description of one gradient list: for each tensor, its scaled
 * FP16 gradient (input), its FP32 unscaled output and its element count.
 * The handle owns a device-resident table that cuts each tensor into chunks
 * of 8192 elements (after a short head chunk up to its first element where
 * input and output are both 32-byte aligned), built once so that each step
 * walks the whole list in a single grid, plus a device workspace: 256 bytes
 * for the step's epilogue words and one fp64 slot per CTA of the unscale
 * grid for the norm form. */
typedef struct gs_tensor_list gs_tensor_list;

/* Build a list on the current device.
 *   grads[i]  -- device pointer to numels[i] FP16 values (scaled gradients)
 *   outs[i]   -- device pointer to numels[i] FP32 values (written by
 *                gs_unscale_check_update)
 *   numels[i] -- >= 0; n_tensors >= 0 (0 gives an empty list)
 * Allocates device memory, uploads the chunk table and clears the
 * workspace, and returns once both are on the device (it synchronises the
 * legacy default stream), so the first step may follow on any stream.  The
 * pointers are captured: the list stays valid while those buffers live.  On
 * error *out is NULL. */
int gs_tensor_list_create(const void* const* grads, void* const* outs, const int64_t* numels,
                          int32_t n_tensors, gs_tensor_list** out);

/* Free a list (NULL is accepted).  Synchronises the device first, so it
 * must not be called while the list is in use by a capture. */
int gs_tensor_list_destroy(gs_tensor_list* list);

/* Total element count and chunk count of a list (host values). */
int gs_tensor_list_info(const gs_tensor_list* list, int64_t* total_elems, int64_t* n_chunks);

/* One GradScaler step over the whole list, in one kernel launch:
 *   out_i = fp32(g_i) * fp32(1 / S)   for every element of every tensor,
 *           where S is *scale as it was before this call; written on
 *           skipped steps too (the caller skips the optimizer);
 *   found_inf = 1 if any g_i is Inf or NaN (exponent field all ones, tested
 *           on the scaled FP16 input), else 0;
 *   then, on the device, after every element has been checked:
 *     found_inf: S *= backoff_factor, growth_tracker = 0, *skipped += 1;
 *     otherwise: growth_tracker += 1 and, if growth_tracker >=
 *                growth_interval, S *= growth_factor, growth_tracker = 0.
 * scale, growth_tracker, found_inf: device scalars (fp32, int32, int32);
 * skipped: device int64 or NULL.  The host never reads any of them.
 * growth_interval >= 1; factors finite and > 0.  (PyTorch-style defaults:
 * S0 = 65536, growth 2.0, backoff 0.5, interval 2000; a static scale is
 * growth_factor = backoff_factor = 1.)  Calls that use the same list must
 * be ordered on one stream (the list's workspace is reused each call). */
int gs_unscale_check_update(const gs_tensor_list* list, float* scale, int32_t* growth_tracker,
                            int32_t* found_inf, int64_t* skipped, float growth_factor,
                            float backoff_factor, int32_t growth_interval, void* stream);

/* The same step, also returning the global L2 norm of the unscaled
 * gradients (step 5 of [P3]'s training step clips by it):
 *   *grad_norm = sqrt(sum over every element of out_i^2)  (device fp32)
 * computed in the same pass (no extra traffic): fp32 fused multiply-adds
 * within a chunk of at most 32 terms per thread, compensated fp32 sums
 * across chunks, fp64 beyond; the sum of squares has a relative error below
 * 35 * 2^-24 and is bitwise reproducible on one device.  A step with
 * Inf/NaN gives an Inf/NaN norm. */
int gs_unscale_check_update_norm(const gs_tensor_list* list, float* scale, int32_t* growth_tracker,
                                 int32_t* found_inf, int64_t* skipped, float growth_factor,
                                 float backoff_factor, int32_t growth_interval, float* grad_norm,
                                 void* stream);

/* The same step under a loss-scale policy with hysteresis ([P3] DeepSpeed
 * paragraph: loss_scale_window 1000, hysteresis 2, consecutive_hysteresis
 * false, min_loss_scale 1 -- the pages name the settings; this reading is
 * the library's): on an overflow the step is skipped, the window restarts
 * (growth_tracker = 0) and, while *hysteresis_state > 1, one unit of it is
 * spent and S kept; with one unit left, S = max(S * backoff_factor,
 * min_scale).  A clean step advances the window; a full window
 * (growth_tracker reaching `window`) multiplies S by growth_factor and
 * restores *hysteresis_state to `hysteresis`; with consecutive_hysteresis
 * != 0 it is restored after every clean step instead.  hysteresis_state is
 * a device int32 the caller initialises to `hysteresis`.  hysteresis = 1
 * and min_scale = 0 give exactly gs_unscale_check_update. */
int gs_unscale_check_update_hysteresis(const gs_tensor_list* list, float* scale,
                                       int32_t* growth_tracker, int32_t* hysteresis_state,
                                       int32_t* found_inf, int64_t* skipped, float growth_factor,
                                       float backoff_factor, int32_t window, int32_t hysteresis,
                                       int32_t consecutive_hysteresis, float min_scale,
                                       void* stream);

/* ------------------------------------------------------------------------
 * The consumer of the step ([P3] six-step training step, step 5: clip and
 * update -- apply guardrails, write into FP32 master state, and skip
 * invalid steps; [P5] "Range and precision": FP32 master weights converted
 * to bf16 each step for the forward pass).
 * --------------------------------------------------------------------- */

/* Opaque list of parameters: per tensor, its fp32 master weights (updated
 * in place), an optional bf16 copy (master_bf16 NULL or master_bf16[i]
 * NULL: none) and its fp32 gradients (typically the outs of a
 * gs_tensor_list).  Allocates a device chunk table and returns once it is
 * on the device (it synchronises the legacy default stream). */
typedef struct gs_param_list gs_param_list;
int gs_param_list_create(float* const* master, uint16_t* const* master_bf16,
                         const float* const* grads, const int64_t* numels, int32_t n_tensors,
                         gs_param_list** out);
int gs_param_list_destroy(gs_param_list* list);

/* SGD step on every parameter of the list, one launch:
 *   if *found_inf != 0 (device): nothing is written (the skipped step);
 *   coef = max_norm / *grad_norm if max_norm > 0 and *grad_norm > max_norm,
 *          else 1 (fp32 division);
 *   w = w - lr * (coef * g), each product and the difference rounded to
 *       fp32 separately; bf16 copy = w rounded to nearest even.
 * grad_norm: device fp32 (from gs_unscale_check_update_norm); may be NULL
 * when max_norm <= 0 (no clipping).  Stream-ordered after the step that
 * produced found_inf / grad_norm; nothing is read on the host. */
int gs_master_update_sgd(const gs_param_list* list, float lr, float max_norm,
                         const float* grad_norm, const int32_t* found_inf, void* stream);

/* Checkpoint support: the scaler's whole state is {S, growth_tracker}.
 * get: copies the two device scalars to host variables and waits for the
 *      copy on `stream` (this call synchronises that stream).
 * set: writes host values into the device scalars, stream-ordered
 *      (asynchronous; the values are passed by value, no host buffer is
 *      kept). */
int gs_scaler_state_get(const float* scale, const int32_t* growth_tracker, float* h_scale,
                        int32_t* h_growth_tracker, void* stream);
int gs_scaler_state_set(float* scale, int32_t* growth_tracker, float h_scale,
                        int32_t h_growth_tracker, void* stream);

/* Allocation-free form of gs_unscale_check_update.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory (code running inside an allocator's own callbacks, or in a
 * process whose device memory another runtime has reserved up front), and so
 * cannot call gs_tensor_list_create.
 *   grads / outs / numels / n_tensors -- as for gs_tensor_list_create, given
 *       on every call (nothing is captured); the remaining arguments and the
 *       results are exactly those of gs_unscale_check_update.
 * The chunk table and the epilogue words live in one fixed device array of
 * this library (768 KiB + 256 B per GPU that loads the library, held until
 * the process exits).  Limits: at most 960 tensors and 32768 chunks of 8192
 * elements (268,435,456 elements in total); larger lists return
 * GS_ERR_SHAPE before anything is launched (see gs_noalloc_limits).
 * The call makes no cudaMalloc / cudaFree and allocates nothing; it uses
 * about 62 KB of the calling thread's stack for the tensor table it passes to
 * the GPU.  Its first call in a CUDA context looks up the array's device
 * address there (cudaGetSymbolAddress) and caches it under the context's ID:
 * each device's primary context, the new primary context that follows a
 * cudaDeviceReset, and any context the caller creates has its own copy of the
 * array and makes its own first call.  Make that first call before any
 * stream capture.  Every call in a context shares that context's array, and
 * its contents persist between calls; the call clears what must start at
 * zero itself.  Calls that overlap on the GPU (on different streams, or from
 * different host threads without ordering) race on the array: order them on
 * one stream. */
int gs_unscale_check_update_noalloc(const void* const* grads, void* const* outs,
                                    const int64_t* numels, int32_t n_tensors, float* scale,
                                    int32_t* growth_tracker, int32_t* found_inf, int64_t* skipped,
                                    float growth_factor, float backoff_factor,
                                    int32_t growth_interval, void* stream);

/* The limits of gs_unscale_check_update_noalloc (host values; any pointer
 * may be NULL). */
int gs_noalloc_limits(int32_t* max_tensors, int64_t* max_chunks, int64_t* chunk_elems);

/* ------------------------------------------------------------------------
 * FP8 quantisation with fine-grained scaling ([P5] "FP8 training", the
 * fp8_scaling.py listing: per-block amax, clamp at 1e-12, divide by MAX;
 * quantise x / s with clamp to +-MAX and cast; dequantise by multiplying
 * by s.  [P1] "FP8 needs a finer-grained fix than a single scale factor"
 * and [P4] "The seam": 1x128 tiles for activations, 128x128 blocks for
 * weights.  [P4] "Failure 1": per-tensor current scaling.)
 *
 * For each block B:   amax_B = max |x| over B (a NaN in B makes it NaN)
 *                     s_B    = max(amax_B, 1e-12f) / MAX      (fp32)
 *                     q      = fp8(clamp(x / s_B, -MAX, MAX)) (fp32 x/s,
 *                              round to nearest even)
 * MAX = 448 (E4M3) or 57344 (E5M2).
 * --------------------------------------------------------------------- */

/* Block-scaled quantisation of a row-major [R, C] tensor.
 *   x        -- R*C elements of in_dtype (GS_BF16, GS_F16 or GS_F32)
 *   (block_r, block_c) -- (1, 128): 1x128 tiles along the contiguous
 *               dimension; or (128, 128): square blocks.  R % block_r == 0
 *               and C % block_c == 0, else GS_ERR_SHAPE.
 *   q        -- R*C bytes of FP8 codes (fmt)
 *   scales   -- fp32 [R / block_r, C / block_c], row-major
 * R == 0 or C == 0 is a valid no-op. */
int fp8_quant_block(const void* x, int in_dtype, int64_t R, int64_t C, int32_t block_r,
                    int32_t block_c, int fmt, uint8_t* q, float* scales, void* stream);

/* Bytes of device workspace fp8_quant_tensor needs (independent of n). */
size_t gs_ws_bytes(void);

/* Per-tensor (current) scaling of n elements: one scale for the whole
 * tensor, computed in a first pass over x and used by a second pass, both
 * on the device (the host never reads amax).
 *   scale -- device fp32 [1], written;  ws -- device workspace of at least
 *   gs_ws_bytes() bytes, 4-byte aligned, any contents (fully overwritten).
 * Calls sharing one ws must be ordered on one stream. */
int fp8_quant_tensor(const void* x, int in_dtype, int64_t n, int fmt, uint8_t* q, float* scale,
                     void* ws, void* stream);

/* Per-tensor quantisation with delayed scaling ([P4] "Failure 1": keep a
 * short history of recent max-abs values and derive s from it; [P5] "FP8
 * training" figure: per tensor, delayed, from recent amax).  One pass over
 * x: the scale applied is s = max(max|amax_history|, 1e-12) / MAX (written
 * to *scale_used); q = fp8(clamp(x / s)); then amax(x) is written at
 * amax_history[*history_pos] and *history_pos advances modulo
 * history_len (1..65536).  amax_history (fp32), history_pos (int32) and
 * scale_used are device memory the caller owns and initialises (a zero
 * history gives the floor scale: everything non-tiny saturates on the
 * first step).  ws: >= gs_ws_bytes() bytes of device scratch.  A NaN in the
 * history makes the scale NaN (every code 0x7F) until it leaves the
 * window.  Calls sharing a history or ws must be ordered on one stream. */
int fp8_quant_tensor_delayed(const void* x, int in_dtype, int64_t n, int fmt, uint8_t* q,
                             float* amax_history, int32_t history_len, int32_t* history_pos,
                             float* scale_used, void* ws, void* stream);

/* Dequantise: y = decode(q) * s (fp32 product), stored as fp32 or rounded
 * to nearest-even bfloat16 (out_dtype GS_F32 or GS_BF16).
 * Block shapes: (1, 128) and (128, 128) with scales laid out as written by
 * fp8_quant_block, or (R, C) -- one scale for the whole [R, C] tensor, as
 * written by fp8_quant_tensor (use R = 1, C = n for a flat tensor). */
int fp8_dequant(const uint8_t* q, const float* scales, int64_t R, int64_t C, int32_t block_r,
                int32_t block_c, int fmt, int out_dtype, void* y, void* stream);

/* ------------------------------------------------------------------------
 * MXFP8: one power-of-two scale per 32 consecutive elements ([P5] "FP8
 * training": Blackwell's MX formats keep one scaling factor per 32 elements
 * in hardware).  The pages give only the block size; the scale rule is the
 * OCP Microscaling convention: an E8M0 byte c means 2^(c - 127) (255 is
 * NaN); for each 1x32 block, e = floor(log2(amax)) - emax_elem (8 for E4M3,
 * 15 for E5M2), clamped to [-127, 127], e = -127 for an all-zero block;
 * q = fp8(x * 2^-e), round to nearest even, saturating at +-MAX; a block
 * holding Inf or NaN gets scale 255 and codes 0x7F.
 * --------------------------------------------------------------------- */

/* x: row-major [R, C] of in_dtype (GS_BF16 / GS_F16 / GS_F32), C % 32 == 0
 * (else GS_ERR_SHAPE); q: R*C FP8 codes; scales: R*C/32 E8M0 bytes,
 * row-major [R, C/32].  Buffers 32-byte aligned with 16-bit input take the
 * vectorised path; any element-aligned buffers are accepted. */
int fp8_quant_mx(const void* x, int in_dtype, int64_t R, int64_t C, int fmt, uint8_t* q,
                 uint8_t* scales, void* stream);

/* y = decode(q) * 2^(scale - 127) in fp32, stored as fp32 or rounded to
 * nearest-even bfloat16 (out_dtype GS_F32 / GS_BF16). */
int fp8_dequant_mx(const uint8_t* q, const uint8_t* scales, int64_t R, int64_t C, int fmt,
                   int out_dtype, void* y, void* stream);

/* ------------------------------------------------------------------------
 * The consumer of the block-scaled tiles: an FP8 GEMM whose partial sums are
 * promoted to FP32 every 128 elements of K ([P1] "FP8 needs a
 * finer-grained fix than a single scale factor": the tensor cores'
 * accumulator keeps too few bits, so partial sums move to FP32 registers at
 * intervals; [P5] "FP8 training": promotion every 128 elements, 1x128
 * scales for activations, 128x128 for weights).
 * --------------------------------------------------------------------- */

/* D = A B^T with A = decode(qa) scaled per 1x128 block and B = decode(qb)
 * scaled per 128x128 block:
 *   D[m][n] = sum over kb of sa[m][kb] * sb[n / 128][kb] * P[m][n][kb],
 *   P[m][n][kb] = sum over k in [128 kb, 128 kb + 128) of
 *                 decode(qa[m][k]) * decode(qb[n][k]).
 * P is formed by the tensor cores (fp32 accumulator, order inside a block
 * not specified); the promotion is one fp32 fused multiply-add per block,
 * acc = fma(P, fp32(sa * sb), acc), in increasing kb.
 *   qa: row-major [M, K] codes, sa: row-major [M, K / 128] fp32 (as
 *       fp8_quant_block writes for block (1, 128));
 *   qb: row-major [N, K] codes (the weight stored [out, in]), sb:
 *       row-major [ceil(N / 128), K / 128] fp32 (block (128, 128));
 *   fmt_a, fmt_b: GS_E4M3 or GS_E5M2, the formats of A and of B; they may
 *      differ ([P5] "FP8 training": E4M3 for forward tensors, E5M2 for
 *      gradients, so a backward GEMM multiplies E5M2 by E4M3);
 *   d: row-major [M, N], out_dtype GS_F32 or GS_BF16 (rounded to nearest
 *      even from the fp32 sum).
 * K % 128 == 0, M, N, K < 2^31 and fewer than 2^30 tiles of 128 x 256
 * (else GS_ERR_SHAPE); M and N need not be multiples of 128; K == 0 writes
 * zeros.  qa and qb must be 16-byte
 * aligned (they are read by TMA; else GS_ERR_ARG).  Accuracy against the
 * exact sum: |error| <= (2^-24 * (nkb + 3) + e_blk) * sum over kb of
 * |sa sb| sum over k |a b|, e_blk being the tensor cores' relative
 * accumulation error within one block.  A wait that runs out records
 * GS_ERR_TIMEOUT (gs_device_status) and leaves d unspecified. */
int fp8_gemm_block_scaled(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                          int64_t M, int64_t N, int64_t K, int fmt_a, int fmt_b, int out_dtype,
                          void* d, void* stream);

/* ------------------------------------------------------------------------
 * Diagnostics.
 * --------------------------------------------------------------------- */

/* Reads and clears the device status word of the current device
 * (GS_OK or GS_ERR_TIMEOUT recorded by a kernel that gave up waiting).
 * Synchronises `stream`. */
int gs_device_status(int32_t* h_status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* GSFP8_H */
