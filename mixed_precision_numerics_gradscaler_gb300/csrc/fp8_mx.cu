// fp8_mx.cu -- MXFP8: FP8 elements with one power-of-two scale per 32
// consecutive elements ("Mixed precision and FP8 training", section "FP8
// training": Blackwell's MX formats keep one scaling factor per 32 elements
// in hardware).  The scale is an E8M0 byte (2^(code - 127), 255 = NaN) with
// shared exponent e = floor(log2(amax)) - emax_elem (8 for E4M3, 15 for
// E5M2) clamped to [-127, 127]; an all-zero block takes e = -127; a block
// holding Inf or NaN gets scale 255 and codes 0x7F.  Elements are cast as
// fp8(x * 2^-e): scaling by a power of two is exact (or rounds once where
// the product leaves the normal range), so x * 2^-e is the IEEE quotient
// x / 2^e.
//
// Layout: one lane per 32-element block -- two 32-byte loads (16-bit input;
// FP32 input takes two lanes per block, quant_mx_f32_v8),
// amax on magnitude bit patterns, the exponent read from the amax's fp32
// exponent field, one 32-byte store of 32 codes and one scale byte (a warp
// writes 32 consecutive scale bytes).  HBM-bound: 2 + 1 + 1/32 bytes per
// element for quantise, 1 + 1/32 + 2 for dequantise to bf16.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gs_device.cuh"
#include "gs_quant.cuh"
#include "gs_internal.h"

namespace gs {

constexpr int kMxThreads = 256;

template <int FMT>
struct MxEmax;
template <>
struct MxEmax<GS_E4M3> {
  static constexpr int value = 8;
};
template <>
struct MxEmax<GS_E5M2> {
  static constexpr int value = 15;
};

// floor(log2(a)) for a finite a > 0 given as fp32 bits (normal or subnormal).
__device__ __forceinline__ int floor_log2_bits(uint32_t bits) {
  return bits >= 0x00800000u ? (int)(bits >> 23) - 127 : (31 - __clz((int)bits)) - 149;
}

// E8M0 code of a block whose finite amax has fp32 bits abits.
template <int FMT>
__device__ __forceinline__ int mx_code(uint32_t abits) {
  if (abits == 0) return 0;
  int e = floor_log2_bits(abits) - MxEmax<FMT>::value;
  e = e < -127 ? -127 : (e > 127 ? 127 : e);
  return e + 127;
}

// 2^(127 - code) as fp32: the element multiplier.  For finite inputs the
// code is at most 127 + 119, so the result is a normal number.
__device__ __forceinline__ float mx_inv_scale(int code) {
  return __uint_as_float((uint32_t)(254 - code) << 23);
}

// 2^(code - 127) as fp32 (code 0 is the subnormal 2^-127), NaN for 255.
__device__ __forceinline__ float mx_scale(uint32_t code) {
  if (code == 255u) return __uint_as_float(0x7FC00000u);
  if (code == 0u) return __uint_as_float(0x00400000u);
  return __uint_as_float(code << 23);
}

template <typename Tag, int FMT>
__global__ void __launch_bounds__(kMxThreads)
    quant_mx_v8(const uint8_t* __restrict__ x, int64_t n_blocks, uint8_t* __restrict__ q,
                uint8_t* __restrict__ scales) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const uint32_t inf16 = std::is_same<Tag, BF16Tag>::value ? 0x7F80u : 0x7C00u;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < n_blocks; b += stride) {
    const V8 a = ld_stream8(x + b * 64), c = ld_stream8(x + b * 64 + 32);
    const uint32_t mm = 0x7FFF7FFFu;
    uint32_t m2 = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) m2 = __vmaxu2(m2, __vmaxu2(a.w[j] & mm, c.w[j] & mm));
    const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    V8 o;
    int code;
    if (m >= inf16) {  // Inf or NaN in the block
      code = 255;
#pragma unroll
      for (int j = 0; j < 8; ++j) o.w[j] = 0x7F7F7F7Fu;
    } else {
      code = mx_code<FMT>(__float_as_uint(mag16_to_float<Tag>(m)));
      const float k = mx_inv_scale(code);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        o.w[j] = cvt_f32x2_fp8x2<FMT>(__fmul_rn(hi16<Tag>(a.w[2 * j]), k),
                                      __fmul_rn(lo16<Tag>(a.w[2 * j]), k)) |
                 (cvt_f32x2_fp8x2<FMT>(__fmul_rn(hi16<Tag>(a.w[2 * j + 1]), k),
                                       __fmul_rn(lo16<Tag>(a.w[2 * j + 1]), k))
                  << 16);
        o.w[4 + j] = cvt_f32x2_fp8x2<FMT>(__fmul_rn(hi16<Tag>(c.w[2 * j]), k),
                                          __fmul_rn(lo16<Tag>(c.w[2 * j]), k)) |
                     (cvt_f32x2_fp8x2<FMT>(__fmul_rn(hi16<Tag>(c.w[2 * j + 1]), k),
                                           __fmul_rn(lo16<Tag>(c.w[2 * j + 1]), k))
                      << 16);
      }
    }
    st_stream8(q + b * 32, o);
    scales[b] = (uint8_t)code;
  }
}

// FP32 input, x 32-byte and q 16-byte aligned: two lanes per 32-element
// block, each with two adjacent 32-byte loads (16 elements); the pair's amax
// by one shuffle; each lane writes 16 codes with one 16-byte store and the
// even lane the scale byte.  Elements scale by the exact power of two on
// f32x2 pairs (each lane an IEEE fp32 multiply).
template <int FMT>
__global__ void __launch_bounds__(kMxThreads)
    quant_mx_f32_v8(const uint8_t* __restrict__ x, int64_t n_blocks, uint8_t* __restrict__ q,
                    uint8_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t n_halves = 2 * n_blocks;
  // warp-uniform loop bound: both lanes of a pair always reach the shuffle
  for (int64_t base = warp * 32; base < n_halves; base += n_warps * 32) {
    const int64_t h = base + lane, b = h >> 1;
    const int part = lane & 1;
    const bool live = h < n_halves;  // false for both lanes of a pair together
    V8 a, c;
    if (live) {
      a = ld_stream8(x + b * 128 + part * 64);
      c = ld_stream8(x + b * 128 + part * 64 + 32);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) a.w[j] = c.w[j] = 0;
    }
    const uint32_t mm = 0x7FFFFFFFu;
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = max(m, max(a.w[j] & mm, c.w[j] & mm));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    uint32_t o[4];
    int code;
    if (m >= 0x7F800000u) {  // Inf or NaN in the block
      code = 255;
#pragma unroll
      for (int j = 0; j < 4; ++j) o[j] = 0x7F7F7F7Fu;
    } else {
      code = mx_code<FMT>(m);
      const float k = mx_inv_scale(code);
      const uint64_t k2 = pk_f32x2(k, k);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const V8& v = j < 2 ? a : c;
        const int w0 = 4 * (j & 1);
        float l0, h0, l1, h1;
        upk_f32x2(mul_f32x2(pk_f32x2(__uint_as_float(v.w[w0]), __uint_as_float(v.w[w0 + 1])), k2),
                  l0, h0);
        upk_f32x2(mul_f32x2(pk_f32x2(__uint_as_float(v.w[w0 + 2]), __uint_as_float(v.w[w0 + 3])), k2),
                  l1, h1);
        o[j] = cvt_f32x2_fp8x2<FMT>(h0, l0) | (cvt_f32x2_fp8x2<FMT>(h1, l1) << 16);
      }
    }
    if (live) {
      *reinterpret_cast<uint4*>(q + b * 32 + part * 16) = make_uint4(o[0], o[1], o[2], o[3]);
      if (part == 0) scales[b] = (uint8_t)code;
    }
  }
}

// Any dtype and alignment: one lane per block, scalar accesses.
template <int DT, int FMT>
__global__ void __launch_bounds__(kMxThreads)
    quant_mx_any(const void* __restrict__ x, int64_t n_blocks, uint8_t* __restrict__ q,
                 uint8_t* __restrict__ scales) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < n_blocks; b += stride) {
    float v[32];
    bool special = false;
    uint32_t amax = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if constexpr (DT == GS_F32) v[i] = reinterpret_cast<const float*>(x)[b * 32 + i];
      else if constexpr (DT == GS_BF16)
        v[i] = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(x)[b * 32 + i] << 16);
      else v[i] = __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(x)[b * 32 + i]));
      const uint32_t mag = __float_as_uint(v[i]) & 0x7FFFFFFFu;
      special |= mag >= 0x7F800000u;
      amax = max(amax, mag);
    }
    const int code = special ? 255 : mx_code<FMT>(amax);
    const float k = special ? 0.0f : mx_inv_scale(code);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      uint32_t c = special ? 0x7F7Fu
                           : cvt_f32x2_fp8x2<FMT>(__fmul_rn(v[i + 1], k), __fmul_rn(v[i], k));
      q[b * 32 + i] = (uint8_t)(c & 0xFFu);
      q[b * 32 + i + 1] = (uint8_t)(c >> 8);
    }
    scales[b] = (uint8_t)code;
  }
}

template <int FMT, int OUT>
__global__ void __launch_bounds__(kMxThreads)
    dequant_mx_v8(const uint8_t* __restrict__ q, const uint8_t* __restrict__ scales,
                  int64_t n_blocks, uint8_t* __restrict__ y) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < n_blocks; b += stride) {
    const V8 c = ld_stream8(q + b * 32);
    const float s = mx_scale(scales[b]);
    float f[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t lo = cvt_fp8x2_f16x2<FMT>((uint16_t)(c.w[i] & 0xFFFFu));
      const uint32_t hi = cvt_fp8x2_f16x2<FMT>((uint16_t)(c.w[i] >> 16));
      f[4 * i + 0] = __fmul_rn(lo_f16(lo), s);
      f[4 * i + 1] = __fmul_rn(hi_f16(lo), s);
      f[4 * i + 2] = __fmul_rn(lo_f16(hi), s);
      f[4 * i + 3] = __fmul_rn(hi_f16(hi), s);
    }
    if constexpr (OUT == GS_F32) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        V8 o;
#pragma unroll
        for (int j = 0; j < 8; ++j) o.w[j] = __float_as_uint(f[8 * k + j]);
        st_stream8(y + b * 128 + 32 * k, o);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        V8 o;
#pragma unroll
        for (int j = 0; j < 8; ++j) o.w[j] = cvt_f32x2_bf16x2(f[16 * k + 2 * j + 1], f[16 * k + 2 * j]);
        st_stream8(y + b * 64 + 32 * k, o);
      }
    }
  }
}

template <int FMT, int OUT>
__global__ void __launch_bounds__(kMxThreads)
    dequant_mx_any(const uint8_t* __restrict__ q, const uint8_t* __restrict__ scales, int64_t n,
                   void* __restrict__ y) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += stride) {
    const float v = __fmul_rn(lo_f16(cvt_fp8x2_f16x2<FMT>(q[e])), mx_scale(scales[e >> 5]));
    if constexpr (OUT == GS_F32) reinterpret_cast<float*>(y)[e] = v;
    else reinterpret_cast<uint16_t*>(y)[e] = (uint16_t)(cvt_f32x2_bf16x2(0.0f, v) & 0xFFFFu);
  }
}

static int64_t mx_grid(int64_t work) {
  int64_t grid = (work + kMxThreads - 1) / kMxThreads;
  const int64_t cap = (int64_t)sm_count() * 64;  // several waves: measured best of 16-128
  return grid > cap ? cap : (grid < 1 ? 1 : grid);
}

template <int DT, int FMT>
static cudaError_t quant_mx_t(const void* x, int64_t nb, uint8_t* q, uint8_t* s, cudaStream_t st) {
  if (DT != GS_F32 && ((uintptr_t)x & 31u) == 0 && ((uintptr_t)q & 31u) == 0) {
    using Tag = typename std::conditional<DT == GS_BF16, BF16Tag, F16Tag>::type;
    quant_mx_v8<Tag, FMT><<<(unsigned)mx_grid(nb), kMxThreads, 0, st>>>(
        reinterpret_cast<const uint8_t*>(x), nb, q, s);
  } else if (DT == GS_F32 && ((uintptr_t)x & 31u) == 0 && ((uintptr_t)q & 15u) == 0) {
    quant_mx_f32_v8<FMT><<<(unsigned)mx_grid(2 * nb), kMxThreads, 0, st>>>(
        reinterpret_cast<const uint8_t*>(x), nb, q, s);
  } else {
    quant_mx_any<DT, FMT><<<(unsigned)mx_grid(nb), kMxThreads, 0, st>>>(x, nb, q, s);
  }
  return cudaGetLastError();
}

cudaError_t launch_quant_mx(const void* x, int dtype, int64_t R, int64_t C, int fmt, uint8_t* q,
                            uint8_t* scales, cudaStream_t st) {
  const int64_t nb = R * (C / 32);
  if (nb == 0) return cudaSuccess;
  if (fmt == GS_E4M3) {
    if (dtype == GS_BF16) return quant_mx_t<GS_BF16, GS_E4M3>(x, nb, q, scales, st);
    if (dtype == GS_F16) return quant_mx_t<GS_F16, GS_E4M3>(x, nb, q, scales, st);
    return quant_mx_t<GS_F32, GS_E4M3>(x, nb, q, scales, st);
  }
  if (dtype == GS_BF16) return quant_mx_t<GS_BF16, GS_E5M2>(x, nb, q, scales, st);
  if (dtype == GS_F16) return quant_mx_t<GS_F16, GS_E5M2>(x, nb, q, scales, st);
  return quant_mx_t<GS_F32, GS_E5M2>(x, nb, q, scales, st);
}

template <int FMT, int OUT>
static cudaError_t dequant_mx_t(const uint8_t* q, const uint8_t* s, int64_t n, void* y,
                                cudaStream_t st) {
  if (((uintptr_t)q & 31u) == 0 && ((uintptr_t)y & 31u) == 0)
    dequant_mx_v8<FMT, OUT><<<(unsigned)mx_grid(n / 32), kMxThreads, 0, st>>>(
        q, s, n / 32, reinterpret_cast<uint8_t*>(y));
  else
    dequant_mx_any<FMT, OUT><<<(unsigned)mx_grid(n), kMxThreads, 0, st>>>(q, s, n, y);
  return cudaGetLastError();
}

cudaError_t launch_dequant_mx(const uint8_t* q, const uint8_t* scales, int64_t R, int64_t C,
                              int fmt, int out_dtype, void* y, cudaStream_t st) {
  const int64_t n = R * C;
  if (n == 0) return cudaSuccess;
  if (fmt == GS_E4M3)
    return out_dtype == GS_F32 ? dequant_mx_t<GS_E4M3, GS_F32>(q, scales, n, y, st)
                               : dequant_mx_t<GS_E4M3, GS_BF16>(q, scales, n, y, st);
  return out_dtype == GS_F32 ? dequant_mx_t<GS_E5M2, GS_F32>(q, scales, n, y, st)
                             : dequant_mx_t<GS_E5M2, GS_BF16>(q, scales, n, y, st);
}

}  // namespace gs
