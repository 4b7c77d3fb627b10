// gs_quant.cuh -- the quantisers' inner step on packed pairs: the two 16-bit
// inputs of a 32-bit word go through the exact quotient together, in f32x2
// arithmetic (one instruction computes both lanes, each an IEEE fp32
// operation rounded to nearest even), and come out as two FP8 codes.
//
// The operations are those of exact_quotient (gs_device.cuh), lane for lane,
// with the negation moved onto the input: with y = -x and nr = -RN(1/s),
//   q = RN(y * nr)          = RN(x * r)
//   n = RN(q * s + y)       = RN(q * s - x)      (the negated residual)
//   q = RN(n * nr + q)      = RN(q - n * r)
// Each line is the same real-number operation as its counterpart, rounded
// once, so every result (signed zeros included) is bit-identical; only the
// sign flips of -x and -n are folded into the inputs, which makes the chain
// free of per-element negations.
#pragma once

#include <stdint.h>

#include <type_traits>

#include "gs_device.cuh"

namespace gs {

// Two fp32 lanes in one 64-bit register: lo = lane 0, hi = lane 1.
__device__ __forceinline__ uint64_t pk_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk_f32x2(uint64_t p, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p));
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// -x for both halves of a word of two 16-bit floats, as exact fp32 values
// (lane 0 from the low half).
template <typename Tag>
__device__ __forceinline__ uint64_t neg_pair(uint32_t w) {
  const uint32_t v = w ^ 0x80008000u;
  if constexpr (std::is_same<Tag, BF16Tag>::value)
    return pk_f32x2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
  else
    return pk_f32x2(lo_f16(v), hi_f16(v));
}

// A block's finite scale s and -RN(1/s), in both lanes.
struct PackedScale {
  uint64_t s2, nr2;
};
__device__ __forceinline__ PackedScale packed_scale(float s, float r) {
  return PackedScale{pk_f32x2(s, s), pk_f32x2(-r, -r)};
}

// Both lanes of exact_quotient<STEPS>(x, s, r), given y = -x.
template <int STEPS>
__device__ __forceinline__ uint64_t exact_quotient_x2(uint64_t y, const PackedScale& ps) {
  uint64_t q = mul_f32x2(y, ps.nr2);
#pragma unroll
  for (int i = 0; i < STEPS; ++i) q = fma_f32x2(fma_f32x2(q, ps.s2, y), ps.nr2, q);
  return q;
}

// Two FP8 codes (low byte from the low half) of a word of two 16-bit inputs,
// for a finite scale.
template <typename Tag, int FMT>
__device__ __forceinline__ uint32_t quant_word_fast(uint32_t w, const PackedScale& ps) {
  float lo, hi;
  upk_f32x2(exact_quotient_x2<QuotSteps<Tag>::value>(neg_pair<Tag>(w), ps), lo, hi);
  return cvt_f32x2_fp8x2<FMT>(hi, lo);
}

// Two FP8 codes of a word for a non-finite scale (a block holding Inf or
// NaN): IEEE division, NaN codes forced to 0x7F.  Out of line: it never runs
// on ordinary data, and keeping it out of the unrolled loops measured faster.
template <typename Tag, int FMT>
__device__ __noinline__ uint32_t quant_word_slow(uint32_t w, float s) {
  return quant_pair<FMT>(hi16<Tag>(w), lo16<Tag>(w), s, 0.0f, false);
}

// NW words of 16-bit pairs -> NW / 2 words of four FP8 codes each, in
// order.  The scale's finiteness is tested once for all of them.
template <typename Tag, int FMT, int NW>
__device__ __forceinline__ void quant_words(const uint32_t* in, uint32_t* out, float s, float r) {
  static_assert(NW % 2 == 0, "words come in pairs");
  if (isfinite(s)) {
    const PackedScale ps = packed_scale(s, r);
#pragma unroll
    for (int j = 0; j < NW / 2; ++j)
      out[j] = quant_word_fast<Tag, FMT>(in[2 * j], ps) |
               (quant_word_fast<Tag, FMT>(in[2 * j + 1], ps) << 16);
  } else {
#pragma unroll
    for (int j = 0; j < NW / 2; ++j)
      out[j] = quant_word_slow<Tag, FMT>(in[2 * j], s) |
               (quant_word_slow<Tag, FMT>(in[2 * j + 1], s) << 16);
  }
}

// quant_words with every input first clamped to [-lim, lim] in fp32, NaN
// kept (for a scale that does not bound the input: delayed scaling).  The
// clamp acts on y = -x, which is the same interval.
template <typename Tag, int FMT>
__device__ __forceinline__ uint32_t quant_word_fast_limited(uint32_t w, const PackedScale& ps,
                                                            float lim) {
  float ylo, yhi, lo, hi;
  upk_f32x2(neg_pair<Tag>(w), ylo, yhi);
  const uint64_t y = pk_f32x2(clamp_keep_nan(ylo, lim), clamp_keep_nan(yhi, lim));
  upk_f32x2(exact_quotient_x2<QuotSteps<Tag>::value>(y, ps), lo, hi);
  return cvt_f32x2_fp8x2<FMT>(hi, lo);
}
template <typename Tag, int FMT, int NW>
__device__ __forceinline__ void quant_words_limited(const uint32_t* in, uint32_t* out, float s,
                                                    float r, float lim) {
  static_assert(NW % 2 == 0, "words come in pairs");
  if (isfinite(s)) {
    const PackedScale ps = packed_scale(s, r);
#pragma unroll
    for (int j = 0; j < NW / 2; ++j)
      out[j] = quant_word_fast_limited<Tag, FMT>(in[2 * j], ps, lim) |
               (quant_word_fast_limited<Tag, FMT>(in[2 * j + 1], ps, lim) << 16);
  } else {
#pragma unroll
    for (int j = 0; j < NW / 2; ++j)
      out[j] = quant_word_slow<Tag, FMT>(in[2 * j], s) |
               (quant_word_slow<Tag, FMT>(in[2 * j + 1], s) << 16);
  }
}

// ---- FP32 inputs ---------------------------------------------------------------
// Two FP8 codes (low byte from x0) of two fp32 inputs given as bit patterns,
// for a finite scale: exact_quotient<2> on both lanes, -x by the sign bit.
template <int FMT>
__device__ __forceinline__ uint32_t quant_f32_pair_fast(uint32_t x0, uint32_t x1,
                                                        const PackedScale& ps) {
  float lo, hi;
  upk_f32x2(exact_quotient_x2<2>(pk_f32x2(__uint_as_float(x0 ^ 0x80000000u),
                                          __uint_as_float(x1 ^ 0x80000000u)),
                                 ps),
            lo, hi);
  return cvt_f32x2_fp8x2<FMT>(hi, lo);
}
template <int FMT>
__device__ __noinline__ uint32_t quant_f32_pair_slow(uint32_t x0, uint32_t x1, float s) {
  return quant_pair<FMT>(__uint_as_float(x1), __uint_as_float(x0), s, 0.0f, false);
}

// NW fp32 words -> NW / 4 words of four FP8 codes each, in order.
template <int FMT, int NW>
__device__ __forceinline__ void quant_words_f32(const uint32_t* in, uint32_t* out, float s,
                                                float r) {
  static_assert(NW % 4 == 0, "four fp32 words per code word");
  if (isfinite(s)) {
    const PackedScale ps = packed_scale(s, r);
#pragma unroll
    for (int j = 0; j < NW / 4; ++j)
      out[j] = quant_f32_pair_fast<FMT>(in[4 * j], in[4 * j + 1], ps) |
               (quant_f32_pair_fast<FMT>(in[4 * j + 2], in[4 * j + 3], ps) << 16);
  } else {
#pragma unroll
    for (int j = 0; j < NW / 4; ++j)
      out[j] = quant_f32_pair_slow<FMT>(in[4 * j], in[4 * j + 1], s) |
               (quant_f32_pair_slow<FMT>(in[4 * j + 2], in[4 * j + 3], s) << 16);
  }
}

// quant_words_f32 with every input first clamped to [-lim, lim], NaN kept.
template <int FMT, int NW>
__device__ __forceinline__ void quant_words_f32_limited(const uint32_t* in, uint32_t* out, float s,
                                                        float r, float lim) {
  uint32_t c[NW];
#pragma unroll
  for (int j = 0; j < NW; ++j) c[j] = __float_as_uint(clamp_keep_nan(__uint_as_float(in[j]), lim));
  quant_words_f32<FMT, NW>(c, out, s, r);
}

}  // namespace gs
