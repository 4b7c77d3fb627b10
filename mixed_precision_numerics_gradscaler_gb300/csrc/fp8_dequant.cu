// fp8_dequant.cu -- y = decode(q) * s ("Why FP8 training is stable",
// "Failure 1": multiply by s on the way out; "Mixed precision and FP8
// training", section "FP8 training": the listing's quant returns
// cast(...).float() * scale).  decode is exact (every E4M3 / E5M2 value is
// an FP16 value: cvt.rn.f16x2.{e4m3x2,e5m2x2}); the product is one fp32
// rounding; the BF16 form rounds that product to nearest even.
//
// dequant_v8 (32-byte aligned codes and output): one thread handles 32
// codes (one 32-byte load) -> 128 B of fp32 or 64 B of bf16 in 32-byte
// stores; dequant_v (16-byte aligned): 16 codes per thread; dequant_any:
// one element per thread.  Scale lookup: 1x128 -> scales[e / 128]; 128x128 ->
// scales[(row / 128) * (C / 128) + col / 128]; per-tensor -> scales[0].
#include <cuda_runtime.h>
#include <stdint.h>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {

constexpr int kDeqThreads = 256;
enum { kBlk1x128 = 0, kBlk128x128 = 1, kBlkTensor = 2 };

template <int KIND>
__device__ __forceinline__ float scale_at(const float* scales, int64_t e, int64_t C) {
  if constexpr (KIND == kBlk1x128) return scales[e >> 7];
  else if constexpr (KIND == kBlk128x128) return scales[(e / C >> 7) * (C >> 7) + ((e % C) >> 7)];
  else return scales[0];
}

template <int FMT>
__device__ __forceinline__ float2 decode2(uint32_t codes16) {
  const uint32_t h2 = cvt_fp8x2_f16x2<FMT>((uint16_t)codes16);
  return make_float2(lo_f16(h2), hi_f16(h2));
}

template <int KIND, int FMT, int OUT>
__global__ void __launch_bounds__(kDeqThreads)
    dequant_v(const uint4* __restrict__ q, const float* __restrict__ scales, int64_t n16, int64_t C,
              void* __restrict__ y) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n16; v += stride) {
    const uint4 c = ld_stream(q + v);
    const float s = scale_at<KIND>(scales, v * 16, C);
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    float f[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = decode2<FMT>(w[i] & 0xFFFFu), b = decode2<FMT>(w[i] >> 16);
      f[4 * i + 0] = __fmul_rn(a.x, s);
      f[4 * i + 1] = __fmul_rn(a.y, s);
      f[4 * i + 2] = __fmul_rn(b.x, s);
      f[4 * i + 3] = __fmul_rn(b.y, s);
    }
    if constexpr (OUT == GS_F32) {
      uint4* yo = reinterpret_cast<uint4*>(y) + 4 * v;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        st_stream(yo + i, make_uint4(__float_as_uint(f[4 * i]), __float_as_uint(f[4 * i + 1]),
                                     __float_as_uint(f[4 * i + 2]), __float_as_uint(f[4 * i + 3])));
    } else {
      uint4* yo = reinterpret_cast<uint4*>(y) + 2 * v;
#pragma unroll
      for (int i = 0; i < 2; ++i)
        st_stream(yo + i, make_uint4(cvt_f32x2_bf16x2(f[8 * i + 1], f[8 * i + 0]),
                                     cvt_f32x2_bf16x2(f[8 * i + 3], f[8 * i + 2]),
                                     cvt_f32x2_bf16x2(f[8 * i + 5], f[8 * i + 4]),
                                     cvt_f32x2_bf16x2(f[8 * i + 7], f[8 * i + 6])));
    }
  }
}

// 32 codes per thread (one 32-byte load) -> 32 outputs (two or four 32-byte
// stores); the 32 elements share one scale for every block shape (32 | 128).
template <int KIND, int FMT, int OUT>
__global__ void __launch_bounds__(kDeqThreads)
    dequant_v8(const uint8_t* __restrict__ q, const float* __restrict__ scales, int64_t n32,
               int64_t C, uint8_t* __restrict__ y) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n32; v += stride) {
    const V8 c = ld_stream8(q + 32 * v);
    const float s = scale_at<KIND>(scales, v * 32, C);
    float f[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 a = decode2<FMT>(c.w[i] & 0xFFFFu), b = decode2<FMT>(c.w[i] >> 16);
      f[4 * i + 0] = __fmul_rn(a.x, s);
      f[4 * i + 1] = __fmul_rn(a.y, s);
      f[4 * i + 2] = __fmul_rn(b.x, s);
      f[4 * i + 3] = __fmul_rn(b.y, s);
    }
    if constexpr (OUT == GS_F32) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        V8 o;
#pragma unroll
        for (int j = 0; j < 8; ++j) o.w[j] = __float_as_uint(f[8 * k + j]);
        st_stream8(y + 128 * v + 32 * k, o);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        V8 o;
#pragma unroll
        for (int j = 0; j < 8; ++j) o.w[j] = cvt_f32x2_bf16x2(f[16 * k + 2 * j + 1], f[16 * k + 2 * j]);
        st_stream8(y + 64 * v + 32 * k, o);
      }
    }
  }
}

// Element-wise path for any alignment and for the ragged tail.
template <int KIND, int FMT, int OUT>
__global__ void __launch_bounds__(kDeqThreads)
    dequant_any(const uint8_t* __restrict__ q, const float* __restrict__ scales, int64_t start,
                int64_t n, int64_t C, void* __restrict__ y) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = start + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += stride) {
    const float v = __fmul_rn(decode2<FMT>(q[e]).x, scale_at<KIND>(scales, e, C));
    if constexpr (OUT == GS_F32) reinterpret_cast<float*>(y)[e] = v;
    else reinterpret_cast<uint16_t*>(y)[e] = (uint16_t)(cvt_f32x2_bf16x2(0.0f, v) & 0xFFFFu);
  }
}

template <int KIND, int FMT, int OUT>
static cudaError_t dequant_t(const uint8_t* q, const float* scales, int64_t R, int64_t C, void* y,
                             cudaStream_t st) {
  const int64_t n = R * C;
  const int64_t cap = (int64_t)sm_count() * 8;
  const size_t ysz = OUT == GS_F32 ? 4 : 2;
  const bool vec = ((uintptr_t)q & 15u) == 0 && ((uintptr_t)y & 15u) == 0;
  const bool vec8 = ((uintptr_t)q & 31u) == 0 && ((uintptr_t)y & 31u) == 0;
  int64_t done = 0;
  if (vec8 && n >= 32) {
    const int64_t n32 = n / 32;
    int64_t grid = (n32 + kDeqThreads - 1) / kDeqThreads;
    const int64_t cap8 = (int64_t)sm_count() * 64;  // several waves: measured best of 32-128
    if (grid > cap8) grid = cap8;
    dequant_v8<KIND, FMT, OUT><<<(unsigned)grid, kDeqThreads, 0, st>>>(
        q, scales, n32, C, reinterpret_cast<uint8_t*>(y));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    done = n32 * 32;
  } else if (vec && n >= 16) {
    const int64_t n16 = n / 16;
    int64_t grid = (n16 + kDeqThreads - 1) / kDeqThreads;
    if (grid > cap) grid = cap;
    dequant_v<KIND, FMT, OUT><<<(unsigned)grid, kDeqThreads, 0, st>>>(
        reinterpret_cast<const uint4*>(q), scales, n16, C, y);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    done = n16 * 16;
  }
  (void)ysz;
  if (done < n) {
    int64_t grid = (n - done + kDeqThreads - 1) / kDeqThreads;
    if (grid > cap) grid = cap;
    dequant_any<KIND, FMT, OUT><<<(unsigned)grid, kDeqThreads, 0, st>>>(q, scales, done, n, C, y);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

template <int KIND>
static cudaError_t dequant_k(const uint8_t* q, const float* scales, int64_t R, int64_t C, int fmt,
                             int out, void* y, cudaStream_t st) {
  if (fmt == GS_E4M3)
    return out == GS_F32 ? dequant_t<KIND, GS_E4M3, GS_F32>(q, scales, R, C, y, st)
                         : dequant_t<KIND, GS_E4M3, GS_BF16>(q, scales, R, C, y, st);
  return out == GS_F32 ? dequant_t<KIND, GS_E5M2, GS_F32>(q, scales, R, C, y, st)
                       : dequant_t<KIND, GS_E5M2, GS_BF16>(q, scales, R, C, y, st);
}

cudaError_t launch_dequant(const uint8_t* q, const float* scales, int64_t R, int64_t C,
                           int block_r, int block_c, int fmt, int out_dtype, void* y,
                           cudaStream_t st) {
  if (R == 0 || C == 0) return cudaSuccess;
  if ((int64_t)block_r == R && (int64_t)block_c == C)
    return dequant_k<kBlkTensor>(q, scales, R, C, fmt, out_dtype, y, st);
  if (block_r == 1) return dequant_k<kBlk1x128>(q, scales, R, C, fmt, out_dtype, y, st);
  return dequant_k<kBlk128x128>(q, scales, R, C, fmt, out_dtype, y, st);
}

}  // namespace gs
