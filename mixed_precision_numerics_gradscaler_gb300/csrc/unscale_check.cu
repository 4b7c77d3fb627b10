// unscale_check.cu -- one GradScaler step over a whole gradient list in a
// single launch ("Loss scaling, FP8, and the failure that never crashes",
// section "Loss scaling, derived from the chain rule you already have",
// and its SimpleGradScaler listing; "Numerical Precision, Mixed Precision,
// and Loss Scaling", GradScaler defaults paragraph and steps 4 and 6 of its
// training step):
//   out = fp32(g) * fp32(1/S) for every element of every tensor,
//   found_inf = any scaled FP16 input with an all-ones exponent field,
//   then S / growth tracker updated on the device by the last CTA to finish.
// Optionally (step 5's clipping needs it) the same pass returns the global
// L2 norm of the unscaled gradients.
//
// Layout: an oversubscribed grid (kUnscaleCtasPerSm CTAs per SM, several waves of
// resident CTAs) walks the list's chunk table grid-stride.  A full 8192-
// element chunk is one pass of a 256-thread CTA: each thread issues two
// 32-byte loads (16 FP16 each) and four 32-byte stores (8 FP32 each).
// Chunks that are short or not 32-byte aligned take a 16-byte path with a
// scalar head and tail.  HBM-bound: 6 bytes per element (2 read + 4
// written).
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {

constexpr int kUnscaleThreads = 256;
constexpr int kUnscaleUnroll = 4;
static_assert(kChunkElems == 2 * 16 * kUnscaleThreads, "one pass of v8 pairs per chunk");

// 0xFFFF in each 16-bit lane whose exponent field is all ones (Inf / NaN).
__device__ __forceinline__ uint32_t nonfinite2(uint32_t w) {
  return __vcmpeq2(w & 0x7C007C00u, 0x7C007C00u);
}

// Sum of squares of the unscaled values, accumulated in fp32 within a
// chunk (at most 32 terms per thread), only in the NORM form.
template <bool NORM>
__device__ __forceinline__ void sq_acc(float& acc, float v) {
  if constexpr (NORM) acc = __fmaf_rn(v, v, acc);
}

template <bool NORM>
__device__ __forceinline__ void unscale8(uint4 v, float inv, uint4* out, uint32_t& bad, float& acc) {
  bad |= nonfinite2(v.x) | nonfinite2(v.y) | nonfinite2(v.z) | nonfinite2(v.w);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float f[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __fmul_rn(lo_f16(w[j]), inv);
    f[2 * j + 1] = __fmul_rn(hi_f16(w[j]), inv);
    sq_acc<NORM>(acc, f[2 * j]);
    sq_acc<NORM>(acc, f[2 * j + 1]);
  }
  st_stream(out, make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                            __float_as_uint(f[3])));
  st_stream(out + 1, make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]),
                                __float_as_uint(f[6]), __float_as_uint(f[7])));
}

template <bool NORM>
__device__ __forceinline__ void unscale1(const uint16_t* in, float* out, int64_t i, float inv,
                                         uint32_t& bad, float& acc) {
  const uint32_t h = in[i];
  bad |= ((h & 0x7C00u) == 0x7C00u);
  const float f = __fmul_rn(__half2float(__ushort_as_half((unsigned short)h)), inv);
  sq_acc<NORM>(acc, f);
  out[i] = f;
}

// Any chunk: 16-byte vectors between a scalar head and tail.
template <bool NORM>
__device__ __forceinline__ uint32_t unscale_chunk(const Chunk ch, float inv, float& acc) {
  const uint16_t* in = ch.in;
  float* out = ch.out;
  const int64_t n = ch.n;
  uint32_t bad = 0;
  // Scalar head until the input is 16-byte aligned; the vector body also
  // needs the output 16-byte aligned at the same element, else all scalar.
  int64_t head = (int64_t)(((16u - ((uint32_t)(uintptr_t)in & 15u)) & 15u) >> 1);
  if (head > n) head = n;
  if ((((uintptr_t)(out + head)) & 15u) != 0) head = n;
  for (int64_t i = threadIdx.x; i < head; i += blockDim.x) unscale1<NORM>(in, out, i, inv, bad, acc);
  const int64_t nv = (n - head) >> 3;
  const uint4* in8 = reinterpret_cast<const uint4*>(in + head);
  uint4* out4 = reinterpret_cast<uint4*>(out + head);
  int64_t v = threadIdx.x;
  for (; v + (kUnscaleUnroll - 1) * (int64_t)blockDim.x < nv; v += kUnscaleUnroll * blockDim.x) {
    uint4 r[kUnscaleUnroll];
#pragma unroll
    for (int u = 0; u < kUnscaleUnroll; ++u) r[u] = ld_stream(in8 + v + u * blockDim.x);
#pragma unroll
    for (int u = 0; u < kUnscaleUnroll; ++u)
      unscale8<NORM>(r[u], inv, out4 + 2 * (v + u * blockDim.x), bad, acc);
  }
  for (; v < nv; v += blockDim.x) unscale8<NORM>(ld_stream(in8 + v), inv, out4 + 2 * v, bad, acc);
  for (int64_t i = head + nv * 8 + threadIdx.x; i < n; i += blockDim.x)
    unscale1<NORM>(in, out, i, inv, bad, acc);
  return bad;
}

// 16 FP16 -> 16 FP32 (two 32-byte stores).
template <bool NORM>
__device__ __forceinline__ void unscale16(const V8& v, float inv, uint8_t* out, uint32_t& bad,
                                          float& acc) {
  V8 a, b;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    bad |= nonfinite2(v.w[j]) | nonfinite2(v.w[j + 4]);
    const float f0 = __fmul_rn(lo_f16(v.w[j]), inv), f1 = __fmul_rn(hi_f16(v.w[j]), inv);
    const float f2 = __fmul_rn(lo_f16(v.w[j + 4]), inv), f3 = __fmul_rn(hi_f16(v.w[j + 4]), inv);
    sq_acc<NORM>(acc, f0);
    sq_acc<NORM>(acc, f1);
    sq_acc<NORM>(acc, f2);
    sq_acc<NORM>(acc, f3);
    a.w[2 * j] = __float_as_uint(f0);
    a.w[2 * j + 1] = __float_as_uint(f1);
    b.w[2 * j] = __float_as_uint(f2);
    b.w[2 * j + 1] = __float_as_uint(f3);
  }
  st_stream8(out, a);
  st_stream8(out + 32, b);
}

// Full, 32-byte-aligned chunk: two loads in flight per thread, then stores.
template <bool NORM>
__device__ __forceinline__ uint32_t unscale_chunk_full(const Chunk ch, float inv, float& acc) {
  const uint8_t* in = reinterpret_cast<const uint8_t*>(ch.in);
  uint8_t* out = reinterpret_cast<uint8_t*>(ch.out);
  const int v0 = threadIdx.x, v1 = threadIdx.x + kUnscaleThreads;
  const V8 a = ld_stream8(in + 32 * v0);
  const V8 b = ld_stream8(in + 32 * v1);
  uint32_t bad = 0;
  unscale16<NORM>(a, inv, out + 64 * v0, bad, acc);
  unscale16<NORM>(b, inv, out + 64 * v1, bad, acc);
  return bad;
}

// With NORM the kernel also returns sqrt(sum of squares) of every unscaled
// value: fp32 fused multiply-adds within a chunk (at most 32 terms per
// thread), Kahan-compensated fp32 sums across a thread's chunks (GB300's
// fp64 rate is far below its fp32 rate, so fp64 stays out of the loop),
// fp64 from the thread total on: across the CTA, one slot per CTA, and the
// last CTA adds the slots in a fixed order.  Deterministic for a given grid; the
// sum of squares carries a relative error below 35 * 2^-24 (all terms are
// non-negative: 32 u per chunk, 2 u for the compensated sum, the rest in
// fp64).
template <bool NORM>
__global__ void __launch_bounds__(kUnscaleThreads)
    unscale_check_update_kernel(const Chunk* __restrict__ chunks, int64_t n_chunks, ListWs* ws,
                                float* scale, int32_t* tracker, int32_t* found_out,
                                int64_t* skipped, float growth, float backoff, int32_t interval,
                                ScalerPolicy pol, float* grad_norm, double* norm_slots) {
  // Every CTA reads S before it arrives below; the last CTA to arrive is the
  // only writer, so all CTAs unscale with this step's S.
  // fp32(1/S) as the oracle defines it, (float)(1.0 / (double)S): for every
  // fp32 S this is the correctly rounded fp32 reciprocal (checked over all
  // 2^32 patterns), so no fp64 division is needed.
  const float S = *scale;
  const float inv = __frcp_rn(S);
  uint32_t bad = 0;
  float ksum = 0.0f, kcomp = 0.0f;  // Kahan sum of the chunk sums
  for (int64_t c = blockIdx.x; c < n_chunks; c += gridDim.x) {
    const Chunk ch = chunks[c];
    const bool full = ch.n == kChunkElems && ((((uintptr_t)ch.in) | ((uintptr_t)ch.out)) & 31u) == 0;
    float acc = 0.0f;
    bad |= full ? unscale_chunk_full<NORM>(ch, inv, acc) : unscale_chunk<NORM>(ch, inv, acc);
    if constexpr (NORM) {
      const float y = __fsub_rn(acc, kcomp);
      const float t = __fadd_rn(ksum, y);
      kcomp = __fsub_rn(__fsub_rn(t, ksum), y);
      ksum = t;
    }
  }
  if constexpr (NORM) {
    double sumsq = (double)ksum - (double)kcomp;
    __shared__ double red[kUnscaleThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sumsq += __shfl_xor_sync(0xFFFFFFFFu, sumsq, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sumsq;
    __syncthreads();
    if (threadIdx.x == 0) {
      double t = 0.0;
      for (int w = 0; w < kUnscaleThreads / 32; ++w) t += red[w];
      norm_slots[blockIdx.x] = t;
    }
  }

  const int any_bad = __syncthreads_or(bad != 0);
  double norm_total = 0.0;
  if constexpr (NORM) {
    // The whole last CTA adds the slots (one fp64 add chain per thread over
    // a fixed stride, then a fixed-order tree): a serial chain of dependent
    // fp64 adds in one thread would take longer than the pass itself.
    __shared__ int last;
    __shared__ double red2[kUnscaleThreads / 32];
    if (threadIdx.x == 0) {
      if (any_bad) atomicOr(&ws->found, 1);
      __threadfence();
      last = atomicAdd(&ws->arrived, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    double t = 0.0;
    for (unsigned int b = threadIdx.x; b < gridDim.x; b += blockDim.x) t += __ldcg(norm_slots + b);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
    if ((threadIdx.x & 31) == 0) red2[threadIdx.x >> 5] = t;
    __syncthreads();
    if (threadIdx.x != 0) return;
    for (int w = 0; w < kUnscaleThreads / 32; ++w) norm_total += red2[w];
  } else {
    if (threadIdx.x != 0) return;
    if (any_bad) atomicOr(&ws->found, 1);
    __threadfence();
    const unsigned int prev = atomicAdd(&ws->arrived, 1u);
    if (prev != gridDim.x - 1) return;
    __threadfence();
  }
  // Last CTA, thread 0: every flag (and every norm slot) is in; apply the
  // control loop.
  const int32_t found = atomicOr(&ws->found, 0) != 0;
  float s = *scale;
  int32_t t = *tracker;
  if (pol.hyst == nullptr) {  // GradScaler loop
    if (found) {
      s = __fmul_rn(s, backoff);
      t = 0;
      if (skipped) *skipped += 1;
    } else {
      t += 1;
      if (t >= interval) {
        s = __fmul_rn(s, growth);
        t = 0;
      }
    }
  } else {  // hysteresis policy
    int32_t h = *pol.hyst;
    if (found) {
      if (skipped) *skipped += 1;
      t = 0;
      if (h > 1) {
        h -= 1;
      } else {
        s = __fmul_rn(s, backoff);
        if (s < pol.min_scale) s = pol.min_scale;
      }
    } else {
      t += 1;
      if (pol.consecutive) h = pol.hysteresis;
      if (t >= interval) {
        s = __fmul_rn(s, growth);
        t = 0;
        if (!pol.consecutive) h = pol.hysteresis;
      }
    }
    *pol.hyst = h;
  }
  *scale = s;
  *tracker = t;
  *found_out = found;
  if constexpr (NORM) *grad_norm = (float)__dsqrt_rn(norm_total);
  ws->found = 0;
  ws->arrived = 0;
}

cudaError_t launch_unscale_check_update(const Chunk* d_chunks, int64_t n_chunks, ListWs* ws,
                                        float* scale, int32_t* tracker, int32_t* found,
                                        int64_t* skipped, float growth, float backoff,
                                        int32_t interval, cudaStream_t stream,
                                        ScalerPolicy policy, float* grad_norm,
                                        double* norm_slots) {
  int64_t grid = (int64_t)sm_count() * kUnscaleCtasPerSm;
  if (grid > n_chunks) grid = n_chunks;
  if (grid < 1) grid = 1;
  if (grad_norm)
    unscale_check_update_kernel<true><<<(unsigned)grid, kUnscaleThreads, 0, stream>>>(
        d_chunks, n_chunks, ws, scale, tracker, found, skipped, growth, backoff, interval, policy,
        grad_norm, norm_slots);
  else
    unscale_check_update_kernel<false><<<(unsigned)grid, kUnscaleThreads, 0, stream>>>(
        d_chunks, n_chunks, ws, scale, tracker, found, skipped, growth, backoff, interval, policy,
        nullptr, nullptr);
  return cudaGetLastError();
}

__global__ void set_state_kernel(float* scale, int32_t* tracker, float h_scale, int32_t h_tracker) {
  *scale = h_scale;
  *tracker = h_tracker;
}

cudaError_t launch_set_state(float* scale, int32_t* tracker, float h_scale, int32_t h_tracker,
                             cudaStream_t stream) {
  set_state_kernel<<<1, 1, 0, stream>>>(scale, tracker, h_scale, h_tracker);
  return cudaGetLastError();
}

}  // namespace gs
