// gs_device.cuh -- device-side building blocks shared by the kernels:
// FP8 pack/unpack through the sm_89+ cvt instructions, 16-bit float
// unpacking, the exact fp32 quotient used by the quantiser, and the
// library's device status word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "gsfp8.h"

namespace gs {

// Largest finite magnitudes of the two OCP FP8 encodings ("Numerical
// Precision, Mixed Precision, and Loss Scaling", paragraph on the FP8
// specification).
template <int FMT>
struct Fp8Max;
template <>
struct Fp8Max<GS_E4M3> {
  static constexpr float value = 448.0f;
};
template <>
struct Fp8Max<GS_E5M2> {
  static constexpr float value = 57344.0f;
};

// Floor applied to every block amax before dividing by MAX ("Mixed
// precision and FP8 training", section "FP8 training": clamp(min=1e-12)).
constexpr float kAmaxFloor = 1e-12f;

// Canonical FP8 NaN written for every NaN input.
constexpr uint32_t kFp8NaN = 0x7Fu;

// ---- FP8 conversions ------------------------------------------------------
// cvt.rn.satfinite.{e4m3x2,e5m2x2}.f32 d, a, b: a -> high byte, b -> low
// byte, round to nearest even, magnitudes beyond the format's max (and
// +-Inf) saturate to +-max.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_f32x2_fp8x2(float hi, float lo) {
  uint16_t d;
  if constexpr (FMT == GS_E4M3) {
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  }
  return d;
}

// Two FP8 codes (low byte first) -> two exact f16 values packed in a word.
template <int FMT>
__device__ __forceinline__ uint32_t cvt_fp8x2_f16x2(uint16_t codes) {
  uint32_t d;
  if constexpr (FMT == GS_E4M3) {
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(codes));
  } else {
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(d) : "h"(codes));
  }
  return d;
}

// Two fp32 values -> two bfloat16 (round to nearest even), hi in the high
// half of the word.
__device__ __forceinline__ uint32_t cvt_f32x2_bf16x2(float hi, float lo) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// ---- 16-bit float unpacking (exact) ---------------------------------------
struct BF16Tag {};
struct F16Tag {};

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float lo_f16(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
}
__device__ __forceinline__ float hi_f16(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

template <typename Tag>
__device__ __forceinline__ float lo16(uint32_t w) {
  if constexpr (std::is_same<Tag, BF16Tag>::value) return lo_bf16(w);
  else return lo_f16(w);
}
template <typename Tag>
__device__ __forceinline__ float hi16(uint32_t w) {
  if constexpr (std::is_same<Tag, BF16Tag>::value) return hi_bf16(w);
  else return hi_f16(w);
}

// Magnitude bit pattern of a 16-bit float held in the low 16 bits -> float.
// For both BF16 and FP16, the unsigned order of magnitude patterns is the
// order of |x|, with Inf above every finite value and NaN above Inf, so an
// integer max over patterns is a NaN-propagating amax.
template <typename Tag>
__device__ __forceinline__ float mag16_to_float(uint32_t m) {
  if constexpr (std::is_same<Tag, BF16Tag>::value) return __uint_as_float(m << 16);
  else return __half2float(__ushort_as_half((unsigned short)m));
}

// ---- scale and exact quotient ---------------------------------------------
// s = max(amax, 1e-12) / MAX in fp32; a NaN amax stays NaN.
template <int FMT>
__device__ __forceinline__ float block_scale(float amax) {
  float a = (amax < kAmaxFloor) ? kAmaxFloor : amax;  // false for NaN: NaN kept
  return __fdiv_rn(a, Fp8Max<FMT>::value);
}

// The fp32 quotient x / s as IEEE division rounds it, for finite s > 0
// (normal), from r = RN(1/s) (computed once per block): one product and
// STEPS residual corrections by fused multiply-add (Markstein's theorem,
// P. Markstein, "IA-64 and Elementary Functions", 2000; Muller et al.,
// "Handbook of Floating-Point Arithmetic", ch. 4: once the estimate is
// within one ulp of x / s, one correction with the correctly rounded
// reciprocal returns the correctly rounded quotient).
//   STEPS = 2 (FP32 inputs): the first correction brings the product,
//     which can be 1.5 ulp off, within one ulp; the second is exact by the
//     theorem whenever |x / s| >= 2^-20, where the residuals cannot
//     underflow (s >= 1e-12 / MAX).
//   STEPS = 1 (BF16 / FP16 inputs): checked by exhaustion over every pair
//     of 16-bit patterns (x, amax) with |x| <= amax, for both formats: the
//     result equals the IEEE quotient bit for bit whenever either is
//     >= 2^-20, and has its sign.
// Below 2^-20 both encode to a signed zero in E4M3 and E5M2, so the FP8
// code is that of the IEEE quotient in every case.  The residual is formed
// negated, n = q*s - x, so that x = -0 yields -0 (the plain form x - q*s
// would give +0 - 0 = +0).
template <int STEPS>
__device__ __forceinline__ float exact_quotient(float x, float s, float r) {
  float q = __fmul_rn(x, r);
#pragma unroll
  for (int i = 0; i < STEPS; ++i) {
    const float n = __fmaf_rn(q, s, -x);
    q = __fmaf_rn(-n, r, q);
  }
  return q;
}

// x clamped to [-lim, lim] (lim >= 0), NaN kept (min.NaN / max.NaN return
// NaN when either operand is NaN, where fminf / fmaxf would drop it).
__device__ __forceinline__ float clamp_keep_nan(float x, float lim) {
  float d;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(x), "f"(lim));
  asm("max.NaN.f32 %0, %0, %1;" : "+f"(d) : "f"(-lim));
  return d;
}

// Quantise a pair with a finite scale (fast path) or a non-finite one (a
// block holding Inf or NaN: IEEE division, NaN codes forced to 0x7F).
template <int FMT, int STEPS = 2>
__device__ __forceinline__ uint32_t quant_pair(float hi, float lo, float s, float r,
                                               bool finite_scale) {
  if (finite_scale)
    return cvt_f32x2_fp8x2<FMT>(exact_quotient<STEPS>(hi, s, r), exact_quotient<STEPS>(lo, s, r));
  float qh = __fdiv_rn(hi, s), ql = __fdiv_rn(lo, s);
  uint32_t c = cvt_f32x2_fp8x2<FMT>(qh, ql);
  if (qh != qh) c = (c & 0x00FFu) | (kFp8NaN << 8);
  if (ql != ql) c = (c & 0xFF00u) | kFp8NaN;
  return c;
}

// Correction steps of the exact quotient for an input type (see above).
template <typename Tag>
struct QuotSteps {
  static constexpr int value = 1;
};

// ---- streaming memory access ----------------------------------------------
// 32-byte (256-bit) global accesses, new with sm_100: half the memory
// instructions of 16-byte accesses for the same bytes in flight.
struct V8 {
  uint32_t w[8];
};
__device__ __forceinline__ V8 ld_stream8(const void* p) {
  V8 a;
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(a.w[0]), "=r"(a.w[1]), "=r"(a.w[2]), "=r"(a.w[3]), "=r"(a.w[4]),
                 "=r"(a.w[5]), "=r"(a.w[6]), "=r"(a.w[7])
               : "l"(p));
  return a;
}
__device__ __forceinline__ void st_stream8(void* p, const V8& a) {
  asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p),
               "r"(a.w[0]), "r"(a.w[1]), "r"(a.w[2]), "r"(a.w[3]), "r"(a.w[4]), "r"(a.w[5]),
               "r"(a.w[6]), "r"(a.w[7])
               : "memory");
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_stream(uint4* p, uint4 v) {
  asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_stream(uint2* p, uint2 v) {
  asm volatile("st.global.L1::no_allocate.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y)
               : "memory");
}

}  // namespace gs
