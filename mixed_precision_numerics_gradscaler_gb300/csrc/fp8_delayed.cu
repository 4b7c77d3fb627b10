// fp8_delayed.cu -- per-tensor FP8 quantisation with delayed scaling ("Why
// FP8 training is stable", "Failure 1": keep a short history of recent
// max-abs values and derive s from it; "Mixed precision and FP8 training",
// "FP8 training" figure: per tensor, delayed, from recent amax).
//
// The scale of this step comes from the history, so one pass reads x once:
//   s = max(max|history|, 1e-12) / MAX        (every CTA, from device memory)
//   q = fp8(clamp(x / s))                      (exact quotient, RNE, saturating)
//   partial amax of x per CTA                  (integer max of magnitude bits)
// and a one-CTA kernel then writes amax(x) at history[pos] and advances
// pos.  3 bytes per 16-bit element instead of current scaling's 5.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gs_device.cuh"
#include "gs_quant.cuh"
#include "gs_internal.h"

namespace gs {

constexpr int kDelThreads = 256;

__device__ __forceinline__ uint32_t block_max_u32(uint32_t m, uint32_t* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0;
#pragma unroll
  for (int w = 0; w < kDelThreads / 32; ++w) m = max(m, red[w]);
  __syncthreads();
  return m;
}

// Delayed scaling takes s from past steps, not from x, so x / s can leave
// the fp32 range: a bf16 or fp32 x above FLT_MAX * s, or an infinite x of
// any type, where the IEEE quotient is +-Inf and the clamp to +-MAX makes
// the code +-MAX.  The exact-quotient chain would meet Inf - Inf there and
// return NaN, so x is first clamped to +-L, L = min(2 MAX s, FLT_MAX), in
// fp32: every |x| >= 2 MAX s gives a quotient above 2 MAX, and x = +-FLT_MAX
// gives one of at least MAX (1 - 2^-23) since s <= FLT_MAX / MAX; all of
// these round to +-MAX, while every |x| <= L is left as it is.  The clamp
// keeps NaN (min.NaN / max.NaN), so a NaN input still gives the NaN code.
// A non-finite s (a NaN or Inf in the history) takes the IEEE division,
// which needs no clamp: its limit is +Inf, which leaves x as it is.
template <int FMT>
__device__ __forceinline__ float quotient_limit(float s) {
  return isfinite(s) ? fminf(__fmul_rn(2.0f * Fp8Max<FMT>::value, s), 3.40282347e38f)
                     : __int_as_float(0x7F800000);
}

// Max |h| over the history as an fp32 bit pattern; NaN entries win (their
// magnitude patterns order above every number).
__device__ __forceinline__ uint32_t history_max_bits(const float* history, int hist_len,
                                                     uint32_t* red) {
  uint32_t m = 0;
  for (int i = threadIdx.x; i < hist_len; i += blockDim.x)
    m = max(m, __float_as_uint(history[i]) & 0x7FFFFFFFu);
  return block_max_u32(m, red);
}

// 16-bit input, x 32-byte and q 16-byte aligned: a grid-stride walk over
// 32-byte vectors, two per iteration (a grid apart).  Each thread issues the
// loads of its next iteration before it casts and stores the current one, and
// its first loads before the history reduction, so 128 bytes per thread are
// in flight.  One persistent wave (74 registers, three CTAs per SM):
// measured 6460 GB/s on GB300 against 6300 for the same walk without the
// prefetch at 16 CTAs per SM.
template <typename Tag, int FMT>
__global__ void __launch_bounds__(kDelThreads)
    quant_delayed_v8(const uint8_t* __restrict__ x, int64_t n, uint8_t* __restrict__ q,
                     const float* __restrict__ history, int hist_len, float* scale_used,
                     uint32_t* __restrict__ partials) {
  __shared__ uint32_t red[kDelThreads / 32];
  constexpr int kSteps = QuotSteps<Tag>::value;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  const int64_t nv = n >> 4;  // 16 elements (32 bytes) per vector
  int64_t v = tid;
  bool have = v + nthreads < nv;
  V8 a, b;
  if (have) {
    a = ld_stream8(x + 32 * v);
    b = ld_stream8(x + 32 * (v + nthreads));
  }
  const float s = block_scale<FMT>(__uint_as_float(history_max_bits(history, hist_len, red)));
  const bool fin = isfinite(s);
  const float r = __frcp_rn(s);
  const float lim = quotient_limit<FMT>(s);
  if (blockIdx.x == 0 && threadIdx.x == 0) *scale_used = s;
  const uint32_t mm = 0x7FFF7FFFu;
  uint32_t m2 = 0;
  while (have) {
    const int64_t vn = v + 2 * nthreads;
    const bool have_next = vn + nthreads < nv;
    V8 na, nb;
    if (have_next) {
      na = ld_stream8(x + 32 * vn);
      nb = ld_stream8(x + 32 * (vn + nthreads));
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) na.w[j] = nb.w[j] = 0;
    }
    uint32_t in[16], c[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      m2 = __vmaxu2(m2, __vmaxu2(a.w[j] & mm, b.w[j] & mm));
      in[j] = a.w[j];
      in[8 + j] = b.w[j];
    }
    quant_words_limited<Tag, FMT, 16>(in, c, s, r, lim);
    st_stream(reinterpret_cast<uint4*>(q + 16 * v), make_uint4(c[0], c[1], c[2], c[3]));
    st_stream(reinterpret_cast<uint4*>(q + 16 * (v + nthreads)), make_uint4(c[4], c[5], c[6], c[7]));
    v = vn;
    a = na;
    b = nb;
    have = have_next;
  }
  for (; v < nv; v += nthreads) {  // at most one vector left per thread
    const V8 a1 = ld_stream8(x + 32 * v);
    uint32_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) m2 = __vmaxu2(m2, __vmaxu2(a1.w[2 * j] & mm, a1.w[2 * j + 1] & mm));
    quant_words_limited<Tag, FMT, 8>(a1.w, c, s, r, lim);
    st_stream(reinterpret_cast<uint4*>(q + 16 * v), make_uint4(c[0], c[1], c[2], c[3]));
  }
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
  // ragged tail (n not a multiple of 16)
  const uint16_t* xs = reinterpret_cast<const uint16_t*>(x);
  for (int64_t i = nv * 16 + tid; i < n; i += nthreads) {
    const uint32_t h = xs[i];
    m = max(m, h & 0x7FFFu);
    const float f = std::is_same<Tag, BF16Tag>::value ? __uint_as_float(h << 16)
                                                       : __half2float(__ushort_as_half((unsigned short)h));
    q[i] = (uint8_t)(quant_pair<FMT, kSteps>(0.0f, clamp_keep_nan(f, lim), s, r, fin) & 0xFFu);
  }
  m = block_max_u32(m, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = m;
}

// FP32 input, x 32-byte and q 8-byte aligned: the same walk over 32-byte
// vectors of eight elements (two per iteration, a grid apart), eight codes
// (one 8-byte store) per vector, cast through quant_words_f32.
template <int FMT>
__global__ void __launch_bounds__(kDelThreads)
    quant_delayed_f32_v8(const uint8_t* __restrict__ x, int64_t n, uint8_t* __restrict__ q,
                         const float* __restrict__ history, int hist_len, float* scale_used,
                         uint32_t* __restrict__ partials) {
  __shared__ uint32_t red[kDelThreads / 32];
  const float s = block_scale<FMT>(__uint_as_float(history_max_bits(history, hist_len, red)));
  const bool fin = isfinite(s);
  const float r = __frcp_rn(s);
  const float lim = quotient_limit<FMT>(s);
  if (blockIdx.x == 0 && threadIdx.x == 0) *scale_used = s;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  const int64_t nv = n >> 3;  // 8 elements (32 bytes) per vector
  const uint32_t mm = 0x7FFFFFFFu;
  uint32_t m = 0;
  int64_t v = tid;
  for (; v + nthreads < nv; v += 2 * nthreads) {
    const V8 a = ld_stream8(x + 32 * v), b = ld_stream8(x + 32 * (v + nthreads));
#pragma unroll
    for (int j = 0; j < 8; ++j) m = max(m, max(a.w[j] & mm, b.w[j] & mm));
    uint32_t ca[2], cb[2];
    quant_words_f32_limited<FMT, 8>(a.w, ca, s, r, lim);
    quant_words_f32_limited<FMT, 8>(b.w, cb, s, r, lim);
    st_stream(reinterpret_cast<uint2*>(q + 8 * v), make_uint2(ca[0], ca[1]));
    st_stream(reinterpret_cast<uint2*>(q + 8 * (v + nthreads)), make_uint2(cb[0], cb[1]));
  }
  for (; v < nv; v += nthreads) {
    const V8 a = ld_stream8(x + 32 * v);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = max(m, a.w[j] & mm);
    uint32_t ca[2];
    quant_words_f32_limited<FMT, 8>(a.w, ca, s, r, lim);
    st_stream(reinterpret_cast<uint2*>(q + 8 * v), make_uint2(ca[0], ca[1]));
  }
  // ragged tail (n not a multiple of 8)
  const float* xf = reinterpret_cast<const float*>(x);
  for (int64_t i = nv * 8 + tid; i < n; i += nthreads) {
    const float f = xf[i];
    m = max(m, __float_as_uint(f) & mm);
    q[i] = (uint8_t)(quant_pair<FMT, 2>(0.0f, clamp_keep_nan(f, lim), s, r, fin) & 0xFFu);
  }
  m = block_max_u32(m, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = m;
}

// Any dtype and alignment, element by element.
template <int DT, int FMT>
__global__ void __launch_bounds__(kDelThreads)
    quant_delayed_any(const void* __restrict__ x, int64_t n, uint8_t* __restrict__ q,
                      const float* __restrict__ history, int hist_len, float* scale_used,
                      uint32_t* __restrict__ partials) {
  __shared__ uint32_t red[kDelThreads / 32];
  const float s = block_scale<FMT>(__uint_as_float(history_max_bits(history, hist_len, red)));
  const bool fin = isfinite(s);
  const float r = __frcp_rn(s);
  const float lim = quotient_limit<FMT>(s);
  if (blockIdx.x == 0 && threadIdx.x == 0) *scale_used = s;
  uint32_t m = 0;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += nthreads) {
    float f;
    uint32_t mag;
    if constexpr (DT == GS_F32) {
      f = reinterpret_cast<const float*>(x)[i];
      mag = __float_as_uint(f) & 0x7FFFFFFFu;
    } else {
      const uint32_t h = reinterpret_cast<const uint16_t*>(x)[i];
      f = DT == GS_BF16 ? __uint_as_float(h << 16) : __half2float(__ushort_as_half((unsigned short)h));
      mag = h & 0x7FFFu;
    }
    m = max(m, mag);
    q[i] = (uint8_t)(quant_pair<FMT, 2>(0.0f, clamp_keep_nan(f, lim), s, r, fin) & 0xFFu);
  }
  m = block_max_u32(m, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = m;
}

// One CTA: amax of this step -> history[pos], pos = (pos + 1) % hist_len.
template <int DT>
__global__ void __launch_bounds__(kDelThreads)
    delayed_record(const uint32_t* __restrict__ partials, int n_partials, float* history,
                   int hist_len, int32_t* pos) {
  __shared__ uint32_t red[kDelThreads / 32];
  uint32_t m = 0;
  for (int i = threadIdx.x; i < n_partials; i += blockDim.x) m = max(m, partials[i]);
  m = block_max_u32(m, red);
  if (threadIdx.x == 0) {
    float a;
    if constexpr (DT == GS_F32) a = __uint_as_float(m);
    else if constexpr (DT == GS_BF16) a = __uint_as_float(m << 16);
    else a = __half2float(__ushort_as_half((unsigned short)m));
    int p = *pos;
    p = (p < 0 || p >= hist_len) ? 0 : p;
    history[p] = a;
    *pos = (p + 1) % hist_len;
  }
}

template <int DT, int FMT>
static cudaError_t delayed_t(const void* x, int64_t n, uint8_t* q, float* history, int hist_len,
                             int32_t* pos, float* scale_used, uint32_t* partials, cudaStream_t st) {
  // One CTA per 8192 elements and at most kMaxAmaxBlocks partials; the
  // 16-bit vector kernel runs one persistent wave, the others at most 16
  // CTAs per SM (more than fit at once: CTAs of later waves even out the
  // SMs, measured faster than one persistent wave for those kernels).
  bool vec = false;
  if constexpr (DT != GS_F32) vec = ((uintptr_t)x & 31u) == 0 && ((uintptr_t)q & 15u) == 0;
  else vec = ((uintptr_t)x & 31u) == 0 && ((uintptr_t)q & 7u) == 0;
  using Tag = typename std::conditional<DT == GS_BF16, BF16Tag, F16Tag>::type;
  int64_t grid = (n + kDelThreads * 32 - 1) / (kDelThreads * 32);
  int64_t cap = (int64_t)sm_count() * 16;
  if (vec && DT != GS_F32) {  // the prefetching kernel: one persistent wave
    int occ = 0;
    const cudaError_t e = kernel_blocks_per_sm((const void*)quant_delayed_v8<Tag, FMT>, kDelThreads, 0, &occ);
    if (e != cudaSuccess) return e;
    cap = (int64_t)sm_count() * (occ < 1 ? 1 : occ);
  }
  if (grid > cap) grid = cap;
  if (grid > kMaxAmaxBlocks) grid = kMaxAmaxBlocks;
  if (grid < 1) grid = 1;
  if (vec && DT == GS_F32)
    quant_delayed_f32_v8<FMT><<<(unsigned)grid, kDelThreads, 0, st>>>(
        reinterpret_cast<const uint8_t*>(x), n, q, history, hist_len, scale_used, partials);
  else if (vec)
    quant_delayed_v8<Tag, FMT><<<(unsigned)grid, kDelThreads, 0, st>>>(
        reinterpret_cast<const uint8_t*>(x), n, q, history, hist_len, scale_used, partials);
  else
    quant_delayed_any<DT, FMT><<<(unsigned)grid, kDelThreads, 0, st>>>(x, n, q, history, hist_len,
                                                                       scale_used, partials);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  delayed_record<DT><<<1, kDelThreads, 0, st>>>(partials, (int)grid, history, hist_len, pos);
  return cudaGetLastError();
}

cudaError_t launch_quant_tensor_delayed(const void* x, int dtype, int64_t n, int fmt, uint8_t* q,
                                        float* history, int hist_len, int32_t* pos,
                                        float* scale_used, uint32_t* partials, cudaStream_t st) {
  if (fmt == GS_E4M3) {
    if (dtype == GS_BF16) return delayed_t<GS_BF16, GS_E4M3>(x, n, q, history, hist_len, pos, scale_used, partials, st);
    if (dtype == GS_F16) return delayed_t<GS_F16, GS_E4M3>(x, n, q, history, hist_len, pos, scale_used, partials, st);
    return delayed_t<GS_F32, GS_E4M3>(x, n, q, history, hist_len, pos, scale_used, partials, st);
  }
  if (dtype == GS_BF16) return delayed_t<GS_BF16, GS_E5M2>(x, n, q, history, hist_len, pos, scale_used, partials, st);
  if (dtype == GS_F16) return delayed_t<GS_F16, GS_E5M2>(x, n, q, history, hist_len, pos, scale_used, partials, st);
  return delayed_t<GS_F32, GS_E5M2>(x, n, q, history, hist_len, pos, scale_used, partials, st);
}

}  // namespace gs
