// master_update.cu -- the step after the cast-and-scale pass ("Numerical
// Precision, Mixed Precision, and Loss Scaling", six-step training step,
// step 5: clip and update -- apply guardrails, write into FP32 master
// state, and skip invalid steps; "Mixed precision and FP8 training",
// "Range and precision": FP32 master weights, converted to bf16 each step
// for the forward pass).
//
// One launch over a parameter list's chunk table:
//   if found_inf (device flag): return -- nothing is written, so every
//                                consumer of the step agrees it was skipped;
//   coef = max_norm / norm if 0 < max_norm < norm, else 1   (fp32 division)
//   w    = w - lr * (coef * g)     (three separately rounded fp32 operations)
//   w_bf16 = RNE(w)                (optional)
// HBM-bound: 4 + 4 read, 4 + 2 written = 14 bytes per parameter.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {

constexpr int kMasterThreads = 256;

__device__ __forceinline__ float sgd1(float w, float g, float lr, float coef) {
  return __fsub_rn(w, __fmul_rn(lr, __fmul_rn(coef, g)));
}

__global__ void __launch_bounds__(kMasterThreads)
    master_update_sgd_kernel(const MChunk* __restrict__ chunks, int64_t n_chunks, float lr,
                             float max_norm, const float* grad_norm, const int32_t* found_inf) {
  if (*found_inf) return;  // skipped step: leave the master state untouched
  float coef = 1.0f;
  if (max_norm > 0.0f) {
    const float nrm = *grad_norm;
    if (nrm > max_norm) coef = __fdiv_rn(max_norm, nrm);
  }
  for (int64_t c = blockIdx.x; c < n_chunks; c += gridDim.x) {
    const MChunk ch = chunks[c];
    const bool vec = ((((uintptr_t)ch.w) | ((uintptr_t)ch.g)) & 31u) == 0 &&
                     (ch.w_bf16 == nullptr || (((uintptr_t)ch.w_bf16) & 15u) == 0);
    const int64_t nv = vec ? ch.n >> 3 : 0;
    for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) {
      const V8 w = ld_stream8(ch.w + 8 * v), g = ld_stream8(ch.g + 8 * v);
      V8 o;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        o.w[j] = __float_as_uint(sgd1(__uint_as_float(w.w[j]), __uint_as_float(g.w[j]), lr, coef));
      st_stream8(ch.w + 8 * v, o);
      if (ch.w_bf16)
        st_stream(reinterpret_cast<uint4*>(ch.w_bf16 + 8 * v),
                  make_uint4(cvt_f32x2_bf16x2(__uint_as_float(o.w[1]), __uint_as_float(o.w[0])),
                             cvt_f32x2_bf16x2(__uint_as_float(o.w[3]), __uint_as_float(o.w[2])),
                             cvt_f32x2_bf16x2(__uint_as_float(o.w[5]), __uint_as_float(o.w[4])),
                             cvt_f32x2_bf16x2(__uint_as_float(o.w[7]), __uint_as_float(o.w[6]))));
    }
    for (int64_t i = nv * 8 + threadIdx.x; i < ch.n; i += blockDim.x) {
      const float w = sgd1(ch.w[i], ch.g[i], lr, coef);
      ch.w[i] = w;
      if (ch.w_bf16) ch.w_bf16[i] = (uint16_t)(cvt_f32x2_bf16x2(0.0f, w) & 0xFFFFu);
    }
  }
}

cudaError_t launch_master_update_sgd(const MChunk* d_chunks, int64_t n_chunks, float lr,
                                     float max_norm, const float* grad_norm,
                                     const int32_t* found_inf, cudaStream_t stream) {
  int64_t grid = (int64_t)sm_count() * 64;  // several waves: measured best of 16-128
  if (grid > n_chunks) grid = n_chunks;
  if (grid < 1) grid = 1;
  master_update_sgd_kernel<<<(unsigned)grid, kMasterThreads, 0, stream>>>(
      d_chunks, n_chunks, lr, max_norm, grad_norm, found_inf);
  return cudaGetLastError();
}

}  // namespace gs
