// fp8_quant.cu -- FP8 quantisation with fine-grained scaling ("Mixed
// precision and FP8 training", section "FP8 training": per-block amax,
// clamp at 1e-12, divide by MAX; q = cast(clamp(x / s)); "Loss scaling,
// FP8, and the failure that never crashes", section "FP8 needs a
// finer-grained fix than a single scale factor": 1x128 tiles for
// activations, 128x128 blocks for weights; "Why FP8 training is stable",
// "Failure 1": per-tensor current scaling).
//
// Kernels:
//   quant_1x128_v8x2 -- BF16/FP16 input, 32-byte aligned (the usual case):
//                       one 4-lane group per 1x128 tile, two 32-byte loads
//                       and one 32-byte store of codes per lane, amax by a
//                       2-step shuffle on magnitude bit patterns.
//   quant_1x128_v8   -- same input, 32-byte aligned x but 16-byte codes: one
//                       8-lane group per tile.
//   quant_1x128_v16  -- BF16/FP16 input, 16-byte aligned: one 16-lane group
//                       per 1x128 tile (8 elements per lane), amax by a
//                       4-step shuffle on magnitude bit patterns.
//   quant_1x128_f32_v8 -- FP32 input, 32-byte aligned (codes 16-byte): one
//                       8-lane group per tile, two 32-byte loads per lane.
//   quant_1x128_v32  -- FP32 input, 16-byte aligned: one warp per tile.
//   quant_1x128_any  -- any dtype / alignment: one warp per tile, scalar.
//   quant_128x128_v8 -- BF16/FP16 input, 32-byte aligned (codes 16-byte):
//                       one 512-thread CTA per 128x128 block, the block
//                       held in registers (two 32-byte loads per thread)
//                       and the CTA's next block loading meanwhile;
//                       quant_128x128_f32_v8 the same block walk for FP32
//                       (four loads, codes 8-byte aligned, no prefetch: a
//                       64 KB block per CTA already keeps enough in flight).
//   quant_128x128_v4 -- the same walk for BF16/FP16 input 16-byte aligned
//                       (codes 8-byte): 16-byte loads, four per thread.
//   quant_128x128_any-- any dtype / alignment: one CTA per block, two
//                       passes over the block (the second hits L2).
//   amax_partials + quant_tensor -- the two passes of per-tensor scaling.
// The vector paths cast through quant_words / quant_words_f32
// (gs_quant.cuh): the exact quotient on f32x2 pairs.
// All paths are HBM-bound: 1x128 moves 2 + 1 + 4/128 bytes per BF16 element.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gs_device.cuh"
#include "gs_quant.cuh"
#include "gs_internal.h"

namespace gs {

constexpr int kQuantThreads = 256;
constexpr int kQuantUnroll = 4;

// ---- generic element access (fallback paths) -------------------------------
template <int DT>
__device__ __forceinline__ uint32_t mag_bits(const void* x, int64_t i) {
  if constexpr (DT == GS_F32) return reinterpret_cast<const uint32_t*>(x)[i] & 0x7FFFFFFFu;
  else return reinterpret_cast<const uint16_t*>(x)[i] & 0x7FFFu;
}
template <int DT>
__device__ __forceinline__ float mag_to_float(uint32_t m) {
  if constexpr (DT == GS_F32) return __uint_as_float(m);
  else if constexpr (DT == GS_BF16) return __uint_as_float(m << 16);
  else return __half2float(__ushort_as_half((unsigned short)m));
}
template <int DT>
__device__ __forceinline__ float load_f(const void* x, int64_t i) {
  if constexpr (DT == GS_F32) return reinterpret_cast<const float*>(x)[i];
  else if constexpr (DT == GS_BF16)
    return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(x)[i] << 16);
  else return __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(x)[i]));
}

template <int FMT>
__device__ __forceinline__ uint8_t quant_one(float v, float s, float r, bool fin) {
  return (uint8_t)(quant_pair<FMT>(0.0f, v, s, r, fin) & 0xFFu);
}

__device__ __forceinline__ uint32_t warp_max(uint32_t m) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  return m;
}

// ---- 1x128, 16-bit input, vectorised ---------------------------------------
template <typename Tag, int FMT>
__global__ void __launch_bounds__(kQuantThreads)
    quant_1x128_v16(const uint4* __restrict__ x, int64_t n_tiles, uint2* __restrict__ q,
                    float* __restrict__ scales) {
  const int lane = threadIdx.x & 31, half = lane >> 4, l16 = lane & 15;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t n_pairs = (n_tiles + 1) >> 1;
  // The loop bound is uniform across the warp, so every lane reaches the
  // shuffles; lanes whose tile is past the end load nothing, store nothing.
  for (int64_t p0 = warp; p0 < n_pairs; p0 += n_warps * kQuantUnroll) {
    uint4 v[kQuantUnroll];
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const int64_t t = 2 * (p0 + u * n_warps) + half;
      v[u] = (t < n_tiles) ? ld_stream(x + t * 16 + l16) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const int64_t t = 2 * (p0 + u * n_warps) + half;
      const uint32_t mm = 0x7FFF7FFFu;
      uint32_t m = __vmaxu2(__vmaxu2(v[u].x & mm, v[u].y & mm), __vmaxu2(v[u].z & mm, v[u].w & mm));
      m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      const float s = block_scale<FMT>(mag16_to_float<Tag>(m));
      const float r = __frcp_rn(s);
      const uint32_t in[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint32_t c[2];
      quant_words<Tag, FMT, 4>(in, c, s, r);
      const uint2 o = make_uint2(c[0], c[1]);
      if (t < n_tiles) {
        st_stream(q + t * 16 + l16, o);
        if (l16 == 0) scales[t] = s;
      }
    }
  }
}

// ---- 1x128, 16-bit input, 32-byte vectors: one 8-lane group per tile -------
// Each lane loads 16 elements (32 B); the 8 lanes of a group reduce the tile
// amax with three shuffles and write 16 codes each (one 16-byte store), so a
// warp moves four tiles per slot and keeps two slots in flight.
constexpr int kQ8Unroll = 2;

__device__ __forceinline__ void st_stream16(void* p, uint4 v) {
  asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

template <typename Tag, int FMT>
__global__ void __launch_bounds__(kQuantThreads)
    quant_1x128_v8(const uint8_t* __restrict__ x, int64_t n_tiles, uint8_t* __restrict__ q,
                   float* __restrict__ scales) {
  const int lane = threadIdx.x & 31, grp = lane >> 3, l8 = lane & 7;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t n_slots = (n_tiles + 3) >> 2;
  // uniform loop bound across the warp: every lane reaches the shuffles
  for (int64_t p0 = warp; p0 < n_slots; p0 += n_warps * kQ8Unroll) {
    V8 v[kQ8Unroll];
#pragma unroll
    for (int u = 0; u < kQ8Unroll; ++u) {
      const int64_t t = 4 * (p0 + u * n_warps) + grp;
      if (t < n_tiles) v[u] = ld_stream8(x + t * 256 + l8 * 32);
      else
#pragma unroll
        for (int j = 0; j < 8; ++j) v[u].w[j] = 0;
    }
#pragma unroll
    for (int u = 0; u < kQ8Unroll; ++u) {
      const int64_t t = 4 * (p0 + u * n_warps) + grp;
      const uint32_t mm = 0x7FFF7FFFu;
      uint32_t m = __vmaxu2(__vmaxu2(__vmaxu2(v[u].w[0] & mm, v[u].w[1] & mm),
                                     __vmaxu2(v[u].w[2] & mm, v[u].w[3] & mm)),
                            __vmaxu2(__vmaxu2(v[u].w[4] & mm, v[u].w[5] & mm),
                                     __vmaxu2(v[u].w[6] & mm, v[u].w[7] & mm)));
      m = max(m & 0xFFFFu, m >> 16);
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      const float s = block_scale<FMT>(mag16_to_float<Tag>(m));
      const float r = __frcp_rn(s);
      uint32_t c[4];
      quant_words<Tag, FMT, 8>(v[u].w, c, s, r);
      if (t < n_tiles) {
        st_stream16(q + t * 128 + l8 * 16, make_uint4(c[0], c[1], c[2], c[3]));
        if (l8 == 0) scales[t] = s;
      }
    }
  }
}

// ---- 1x128, 16-bit input: one 4-lane group per tile --------------------------
// Each lane loads 32 elements (two 32-byte loads) of its tile; the 4 lanes
// reduce the tile amax with two shuffles; each lane writes its 32 codes with
// one 32-byte store.  A warp moves eight tiles (2 KB in, 1 KB out) per slot,
// and the per-tile scale and reciprocal are amortised over 32 elements per
// lane.
template <typename Tag, int FMT>
__global__ void __launch_bounds__(kQuantThreads)
    quant_1x128_v8x2(const uint8_t* __restrict__ x, int64_t n_tiles, uint8_t* __restrict__ q,
                     float* __restrict__ scales) {
  const int lane = threadIdx.x & 31, grp = lane >> 2, l4 = lane & 3;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t n_slots = (n_tiles + 7) >> 3;
  // uniform loop bound across the warp: every lane reaches the shuffles
  for (int64_t p0 = warp; p0 < n_slots; p0 += n_warps) {
    const int64_t t = 8 * p0 + grp;
    V8 a, b;
    if (t < n_tiles) {
      a = ld_stream8(x + t * 256 + l4 * 64);
      b = ld_stream8(x + t * 256 + l4 * 64 + 32);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) a.w[j] = b.w[j] = 0;
    }
    const uint32_t mm = 0x7FFF7FFFu;
    uint32_t m2 = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) m2 = __vmaxu2(m2, __vmaxu2(a.w[j] & mm, b.w[j] & mm));
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    const float s = block_scale<FMT>(mag16_to_float<Tag>(m));
    const float r = __frcp_rn(s);
    uint32_t in[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      in[j] = a.w[j];
      in[8 + j] = b.w[j];
    }
    V8 o;
    quant_words<Tag, FMT, 16>(in, o.w, s, r);
    if (t < n_tiles) {
      st_stream8(q + t * 128 + l4 * 32, o);
      if (l4 == 0) scales[t] = s;
    }
  }
}

// ---- 128x128, 16-bit input, direct 32-byte loads -----------------------------
// One 512-thread CTA per 128x128 block at a time, grid-stride over the blocks
// with two CTAs resident per SM.  Thread t loads the 32-byte chunk t mod 8
// of rows t/8 and t/8 + 64 of the block (a warp reads four whole 256-byte
// rows per load instruction), so the block sits in registers, 32 elements per
// thread.  The loads of the CTA's next block are issued before the barrier
// that completes this block's amax, so they are in flight while the block is
// reduced, scaled, cast and stored: each CTA always has one block (32 KB)
// loading.  Block amax: packed magnitude max, warp shuffles, one word per warp
// in shared memory (two sets, alternating by block, so one barrier per block
// suffices), read back by every thread as four 16-byte vectors.  Codes leave
// as two 16-byte stores per thread.  Measured on GB300 (bf16 8192x28672):
// 6700 GB/s, against 6350 for the same walk without the prefetch at three
// CTAs per SM (38 registers) and 5750-6200 for a TMA-staged form with 2-3
// stages of 32 KB per CTA.
constexpr int kQ128Threads = 512;
constexpr int kQ128Warps = kQ128Threads / 32;
constexpr int kQ128RowStep = kQ128Threads / 8;  // 64: rows between a thread's two loads

template <typename Tag, int FMT>
__global__ void __launch_bounds__(kQ128Threads, 2)
    quant_128x128_v8(const uint8_t* __restrict__ x, int64_t nbr, int64_t nbc,
                     uint8_t* __restrict__ q, int64_t C, float* __restrict__ scales) {
  __shared__ __align__(16) uint32_t red[2][kQ128Warps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk = tid & 7, row = tid >> 3;
  const int64_t n_blocks = nbr * nbc;
  if ((int64_t)blockIdx.x >= n_blocks) return;
  const int64_t row_bytes = C * 2;
  // block b = blockIdx.x + k * gridDim.x is (b / nbc, b % nbc); both advance
  // by gridDim.x's quotient and remainder, so the loop divides nothing
  const int64_t step_r = gridDim.x / nbc, step_c = gridDim.x % nbc;
  int64_t br = blockIdx.x / nbc, bc = blockIdx.x % nbc;
  V8 a, c;
  {
    const uint8_t* xb = x + (br * 128 + row) * row_bytes + bc * 256 + chunk * 32;
    a = ld_stream8(xb);
    c = ld_stream8(xb + kQ128RowStep * row_bytes);
  }
  int par = 0;
  for (int64_t b = blockIdx.x; b < n_blocks; b += gridDim.x, par ^= 1) {
    const uint32_t mm = 0x7FFF7FFFu;
    uint32_t m2 = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) m2 = __vmaxu2(m2, __vmaxu2(a.w[j] & mm, c.w[j] & mm));
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) red[par][warp] = m;
    // the next block of this CTA (if any): its loads go out now
    int64_t nbr_next = br + step_r, nbc_next = bc + step_c;
    if (nbc_next >= nbc) {
      nbc_next -= nbc;
      ++nbr_next;
    }
    V8 na, nc;
    if (b + gridDim.x < n_blocks) {
      const uint8_t* xn = x + (nbr_next * 128 + row) * row_bytes + nbc_next * 256 + chunk * 32;
      na = ld_stream8(xn);
      nc = ld_stream8(xn + kQ128RowStep * row_bytes);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) na.w[j] = nc.w[j] = 0;
    }
    __syncthreads();
    {
      const uint4* r4 = reinterpret_cast<const uint4*>(red[par]);
      uint4 v = r4[0];
#pragma unroll
      for (int w = 1; w < kQ128Warps / 4; ++w) {
        const uint4 u = r4[w];
        v = make_uint4(max(v.x, u.x), max(v.y, u.y), max(v.z, u.z), max(v.w, u.w));
      }
      m = max(max(v.x, v.y), max(v.z, v.w));
    }
    const float s = block_scale<FMT>(mag16_to_float<Tag>(m));
    const float r = __frcp_rn(s);
    if (tid == 0) scales[b] = s;
    uint32_t ca[4], cc[4];
    quant_words<Tag, FMT, 8>(a.w, ca, s, r);
    quant_words<Tag, FMT, 8>(c.w, cc, s, r);
    uint8_t* qb = q + (br * 128 + row) * C + bc * 128 + chunk * 16;
    st_stream(reinterpret_cast<uint4*>(qb), make_uint4(ca[0], ca[1], ca[2], ca[3]));
    st_stream(reinterpret_cast<uint4*>(qb + kQ128RowStep * C), make_uint4(cc[0], cc[1], cc[2], cc[3]));
    br = nbr_next;
    bc = nbc_next;
    a = na;
    c = nc;
  }
}

// ---- 128x128, 16-bit input, direct 16-byte loads ----------------------------
// The same block walk as quant_128x128_v8 for x 16-byte aligned and q 8-byte
// aligned: thread t loads the 16-byte chunk t mod 16 of rows t/16 + 32 i,
// i < 4 (a warp reads two whole 256-byte rows per load instruction), 32
// elements per thread, and the loads of the CTA's next block go out before
// the barrier that completes this block's amax.  Codes leave as four 8-byte
// stores per thread.  Measured on GB300 (bf16 8192x28672 at a 16-byte
// offset): 6588 GB/s, against 5320-5756 for a TMA-staged form (a 3-stage ring
// of 32 KB tiles per CTA, 512 threads pulling each tile out of shared memory).
constexpr int kQ128V4RowStep = kQ128Threads / 16;  // 32

template <typename Tag, int FMT>
__global__ void __launch_bounds__(kQ128Threads, 2)
    quant_128x128_v4(const uint8_t* __restrict__ x, int64_t nbr, int64_t nbc,
                     uint8_t* __restrict__ q, int64_t C, float* __restrict__ scales) {
  __shared__ __align__(16) uint32_t red[2][kQ128Warps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk = tid & 15, row = tid >> 4;
  const int64_t n_blocks = nbr * nbc;
  if ((int64_t)blockIdx.x >= n_blocks) return;
  const int64_t row_bytes = C * 2;
  const int64_t step_r = gridDim.x / nbc, step_c = gridDim.x % nbc;
  int64_t br = blockIdx.x / nbc, bc = blockIdx.x % nbc;
  uint4 v[4];
  {
    const uint8_t* xb = x + (br * 128 + row) * row_bytes + bc * 256 + chunk * 16;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      v[i] = ld_stream(reinterpret_cast<const uint4*>(xb + i * kQ128V4RowStep * row_bytes));
  }
  int par = 0;
  for (int64_t b = blockIdx.x; b < n_blocks; b += gridDim.x, par ^= 1) {
    const uint32_t mm = 0x7FFF7FFFu;
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(v[i].x & mm, v[i].y & mm),
                                 __vmaxu2(v[i].z & mm, v[i].w & mm)));
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) red[par][warp] = m;
    int64_t nbr_next = br + step_r, nbc_next = bc + step_c;
    if (nbc_next >= nbc) {
      nbc_next -= nbc;
      ++nbr_next;
    }
    uint4 nv[4];
    if (b + gridDim.x < n_blocks) {
      const uint8_t* xn = x + (nbr_next * 128 + row) * row_bytes + nbc_next * 256 + chunk * 16;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        nv[i] = ld_stream(reinterpret_cast<const uint4*>(xn + i * kQ128V4RowStep * row_bytes));
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) nv[i] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    {
      const uint4* r4 = reinterpret_cast<const uint4*>(red[par]);
      uint4 u = r4[0];
#pragma unroll
      for (int w = 1; w < kQ128Warps / 4; ++w) {
        const uint4 t4 = r4[w];
        u = make_uint4(max(u.x, t4.x), max(u.y, t4.y), max(u.z, t4.z), max(u.w, t4.w));
      }
      m = max(max(u.x, u.y), max(u.z, u.w));
    }
    const float s = block_scale<FMT>(mag16_to_float<Tag>(m));
    const float r = __frcp_rn(s);
    if (tid == 0) scales[b] = s;
    uint32_t in[16], c[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      in[4 * i] = v[i].x;
      in[4 * i + 1] = v[i].y;
      in[4 * i + 2] = v[i].z;
      in[4 * i + 3] = v[i].w;
    }
    quant_words<Tag, FMT, 16>(in, c, s, r);
    uint8_t* qb = q + (br * 128 + row) * C + bc * 128 + chunk * 8;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      st_stream(reinterpret_cast<uint2*>(qb + i * kQ128V4RowStep * C), make_uint2(c[2 * i], c[2 * i + 1]));
    br = nbr_next;
    bc = nbc_next;
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = nv[i];
  }
}


// ---- 128x128, FP32 input, direct 32-byte loads ---------------------------------
// The FP32 form of quant_128x128_v8: a block row is 512 bytes, so thread t
// loads the 32-byte chunk t mod 16 of rows t/16 + 32 i, i < 4 (a warp reads
// two whole rows per load instruction), 32 elements per thread; codes leave
// as four 8-byte stores per thread (a warp writes two 128-byte code rows).
constexpr int kQ128F32RowStep = kQ128Threads / 16;  // 32

template <int FMT>
__global__ void __launch_bounds__(kQ128Threads, 2)
    quant_128x128_f32_v8(const uint8_t* __restrict__ x, int64_t nbr, int64_t nbc,
                         uint8_t* __restrict__ q, int64_t C, float* __restrict__ scales) {
  __shared__ __align__(16) uint32_t red[2][kQ128Warps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk = tid & 15, row = tid >> 4;
  const int64_t n_blocks = nbr * nbc;
  if ((int64_t)blockIdx.x >= n_blocks) return;
  const int64_t row_bytes = C * 4;
  const int64_t step_r = gridDim.x / nbc, step_c = gridDim.x % nbc;
  int64_t br = blockIdx.x / nbc, bc = blockIdx.x % nbc;
  int par = 0;
  for (int64_t b = blockIdx.x; b < n_blocks; b += gridDim.x, par ^= 1) {
    const uint8_t* xb = x + (br * 128 + row) * row_bytes + bc * 512 + chunk * 32;
    V8 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = ld_stream8(xb + i * kQ128F32RowStep * row_bytes);
    const uint32_t mm = 0x7FFFFFFFu;
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) m = max(m, v[i].w[j] & mm);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) red[par][warp] = m;
    __syncthreads();
    {
      const uint4* r4 = reinterpret_cast<const uint4*>(red[par]);
      uint4 u = r4[0];
#pragma unroll
      for (int w = 1; w < kQ128Warps / 4; ++w) {
        const uint4 t4 = r4[w];
        u = make_uint4(max(u.x, t4.x), max(u.y, t4.y), max(u.z, t4.z), max(u.w, t4.w));
      }
      m = max(max(u.x, u.y), max(u.z, u.w));
    }
    const float s = block_scale<FMT>(__uint_as_float(m));
    const float r = __frcp_rn(s);
    if (tid == 0) scales[b] = s;
    uint8_t* qb = q + (br * 128 + row) * C + bc * 128 + chunk * 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t c[2];
      quant_words_f32<FMT, 8>(v[i].w, c, s, r);
      st_stream(reinterpret_cast<uint2*>(qb + i * kQ128F32RowStep * C), make_uint2(c[0], c[1]));
    }
    br += step_r;
    bc += step_c;
    if (bc >= nbc) {
      bc -= nbc;
      ++br;
    }
  }
}

// ---- 1x128, FP32 input, 32-byte aligned: one 8-lane group per tile -----------
// Each lane loads 16 elements (two adjacent 32-byte loads) of its tile, the
// 8 lanes reduce the tile amax (integer max of fp32 magnitude patterns, three
// shuffles), and each lane casts its 16 elements through quant_words_f32 and
// writes one 16-byte store of codes.  A warp moves four tiles (2 KB in,
// 512 B out) per slot.
template <int FMT>
__global__ void __launch_bounds__(kQuantThreads)
    quant_1x128_f32_v8(const uint8_t* __restrict__ x, int64_t n_tiles, uint8_t* __restrict__ q,
                       float* __restrict__ scales) {
  const int lane = threadIdx.x & 31, grp = lane >> 3, l8 = lane & 7;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t n_slots = (n_tiles + 3) >> 2;
  // uniform loop bound across the warp: every lane reaches the shuffles
  for (int64_t p0 = warp; p0 < n_slots; p0 += n_warps) {
    const int64_t t = 4 * p0 + grp;
    V8 a, b;
    if (t < n_tiles) {
      a = ld_stream8(x + t * 512 + l8 * 64);
      b = ld_stream8(x + t * 512 + l8 * 64 + 32);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) a.w[j] = b.w[j] = 0;
    }
    const uint32_t mm = 0x7FFFFFFFu;
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = max(m, max(a.w[j] & mm, b.w[j] & mm));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    const float s = block_scale<FMT>(__uint_as_float(m));
    const float r = __frcp_rn(s);
    uint32_t in[16], c[4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      in[j] = a.w[j];
      in[8 + j] = b.w[j];
    }
    quant_words_f32<FMT, 16>(in, c, s, r);
    if (t < n_tiles) {
      st_stream16(q + t * 128 + l8 * 16, make_uint4(c[0], c[1], c[2], c[3]));
      if (l8 == 0) scales[t] = s;
    }
  }
}

// ---- 1x128, FP32 input, vectorised: one warp per tile ------------------------
template <int FMT>
__global__ void __launch_bounds__(kQuantThreads)
    quant_1x128_v32(const uint4* __restrict__ x, int64_t n_tiles, uint32_t* __restrict__ q,
                    float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t = warp; t < n_tiles; t += n_warps) {
    const uint4 v = ld_stream(x + t * 32 + lane);
    const uint32_t mm = 0x7FFFFFFFu;
    uint32_t m = max(max(v.x & mm, v.y & mm), max(v.z & mm, v.w & mm));
    m = warp_max(m);
    const float s = block_scale<FMT>(__uint_as_float(m));
    const bool fin = isfinite(s);
    const float r = __frcp_rn(s);
    const uint32_t c = quant_pair<FMT>(__uint_as_float(v.y), __uint_as_float(v.x), s, r, fin) |
                       (quant_pair<FMT>(__uint_as_float(v.w), __uint_as_float(v.z), s, r, fin) << 16);
    q[t * 32 + lane] = c;
    if (lane == 0) scales[t] = s;
  }
}

// ---- 1x128, any dtype and alignment ------------------------------------------
template <int DT, int FMT>
__global__ void __launch_bounds__(kQuantThreads)
    quant_1x128_any(const void* __restrict__ x, int64_t n_tiles, uint8_t* __restrict__ q,
                    float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t = warp; t < n_tiles; t += n_warps) {
    const int64_t base = t * 128;
    uint32_t m = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) m = max(m, mag_bits<DT>(x, base + lane + 32 * k));
    m = warp_max(m);
    const float s = block_scale<FMT>(mag_to_float<DT>(m));
    const bool fin = isfinite(s);
    const float r = __frcp_rn(s);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t i = base + lane + 32 * k;
      q[i] = quant_one<FMT>(load_f<DT>(x, i), s, r, fin);
    }
    if (lane == 0) scales[t] = s;
  }
}

// ---- 128x128, any dtype and alignment: one CTA per block --------------------
template <int DT, int FMT>
__global__ void __launch_bounds__(kQuantThreads)
    quant_128x128_any(const void* __restrict__ x, int64_t R, int64_t C, uint8_t* __restrict__ q,
                      float* __restrict__ scales) {
  __shared__ uint32_t red[kQuantThreads / 32];
  __shared__ float s_sh;
  const int64_t nbc = C / 128, n_blocks = (R / 128) * nbc;
  for (int64_t b = blockIdx.x; b < n_blocks; b += gridDim.x) {
    const int64_t r0 = (b / nbc) * 128, c0 = (b % nbc) * 128;
    uint32_t m = 0;
    for (int k = threadIdx.x; k < 128 * 128; k += blockDim.x)
      m = max(m, mag_bits<DT>(x, (r0 + (k >> 7)) * C + c0 + (k & 127)));
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t mm = 0;
      for (int w = 0; w < kQuantThreads / 32; ++w) mm = max(mm, red[w]);
      const float s = block_scale<FMT>(mag_to_float<DT>(mm));
      s_sh = s;
      scales[b] = s;
    }
    __syncthreads();
    const float s = s_sh;
    const bool fin = isfinite(s);
    const float r = __frcp_rn(s);
    for (int k = threadIdx.x; k < 128 * 128; k += blockDim.x) {
      const int64_t i = (r0 + (k >> 7)) * C + c0 + (k & 127);
      q[i] = quant_one<FMT>(load_f<DT>(x, i), s, r, fin);
    }
    __syncthreads();  // red / s_sh are reused by the next block
  }
}

// ---- per-tensor: pass 1, per-CTA amax partials --------------------------------
template <int DT>
__global__ void __launch_bounds__(kQuantThreads)
    amax_partials(const void* __restrict__ x, int64_t n, uint32_t* __restrict__ partials) {
  __shared__ uint32_t red[kQuantThreads / 32];
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  uint32_t m = 0;
  if constexpr (DT != GS_F32) {
    // 16-byte vectors once the pointer is aligned; scalar head and tail.
    const uint16_t* xs = reinterpret_cast<const uint16_t*>(x);
    int64_t head = (int64_t)(((16u - ((uint32_t)(uintptr_t)xs & 15u)) & 15u) >> 1);
    if (head > n) head = n;
    for (int64_t i = tid; i < head; i += nthreads) m = max(m, (uint32_t)(xs[i] & 0x7FFFu));
    const int64_t nv = (n - head) >> 3;
    const uint4* x8 = reinterpret_cast<const uint4*>(xs + head);
    uint32_t m2 = 0;
    const uint32_t mm = 0x7FFF7FFFu;
    int64_t v = tid;
    for (; v + 3 * nthreads < nv; v += 4 * nthreads) {
      uint4 a[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] = ld_stream(x8 + v + u * nthreads);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(a[u].x & mm, a[u].y & mm),
                                   __vmaxu2(a[u].z & mm, a[u].w & mm)));
    }
    for (; v < nv; v += nthreads) {
      const uint4 a = ld_stream(x8 + v);
      m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(a.x & mm, a.y & mm), __vmaxu2(a.z & mm, a.w & mm)));
    }
    m = max(m, max(m2 & 0xFFFFu, m2 >> 16));
    for (int64_t i = head + nv * 8 + tid; i < n; i += nthreads) m = max(m, (uint32_t)(xs[i] & 0x7FFFu));
  } else {
    // 16-byte vectors of four fp32 once the pointer is aligned
    const uint32_t* xs = reinterpret_cast<const uint32_t*>(x);
    int64_t head = (int64_t)(((16u - ((uint32_t)(uintptr_t)xs & 15u)) & 15u) >> 2);
    if (head > n) head = n;
    const uint32_t mm = 0x7FFFFFFFu;
    for (int64_t i = tid; i < head; i += nthreads) m = max(m, xs[i] & mm);
    const int64_t nv = (n - head) >> 2;
    const uint4* x4 = reinterpret_cast<const uint4*>(xs + head);
    int64_t v = tid;
    for (; v + 3 * nthreads < nv; v += 4 * nthreads) {
      uint4 a[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] = ld_stream(x4 + v + u * nthreads);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        m = max(m, max(max(a[u].x & mm, a[u].y & mm), max(a[u].z & mm, a[u].w & mm)));
    }
    for (; v < nv; v += nthreads) {
      const uint4 a = ld_stream(x4 + v);
      m = max(m, max(max(a.x & mm, a.y & mm), max(a.z & mm, a.w & mm)));
    }
    for (int64_t i = head + nv * 4 + tid; i < n; i += nthreads) m = max(m, xs[i] & mm);
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t mm = 0;
    for (int w = 0; w < kQuantThreads / 32; ++w) mm = max(mm, red[w]);
    partials[blockIdx.x] = mm;
  }
}

// ---- per-tensor: pass 2, reduce the partials, quantise ------------------------
// Pass 1 reads x in ascending address order, so when it ends the L2 still
// holds the end of x.  Pass 2 therefore walks the vector body from the
// highest address down: the body is cut into iterations of kQuantThreads x 4
// vectors, CTA c takes the run of kPass2Run consecutive iterations counted
// c runs from the END, and CTAs start roughly in index order, so the first
// ones read what pass 1 left in L2.  Measured on GB300 (bf16 8192x28672,
// E5M2, both passes): 6769 GB/s against 6395 for the ascending grid-stride
// walk at 32 CTAs per SM.  Every CTA first reduces the partials itself.
constexpr int kPass2Run = 2;
constexpr int64_t kPass2It = (int64_t)kQuantThreads * 4;  // vectors per iteration

template <int DT, int FMT>
__global__ void __launch_bounds__(kQuantThreads)
    quant_tensor_pass2(const void* __restrict__ x, int64_t n, uint8_t* __restrict__ q,
                       float* __restrict__ scale_out, const uint32_t* __restrict__ partials,
                       int n_partials) {
  __shared__ uint32_t red[kQuantThreads / 32];
  uint32_t m = 0;
  for (int i = threadIdx.x; i < n_partials; i += blockDim.x) m = max(m, partials[i]);
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0;
#pragma unroll
  for (int w = 0; w < kQuantThreads / 32; ++w) m = max(m, red[w]);
  const float s = block_scale<FMT>(mag_to_float<DT>(m));
  const bool fin = isfinite(s);
  const float r = __frcp_rn(s);
  if (blockIdx.x == 0 && threadIdx.x == 0) *scale_out = s;

  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  if constexpr (DT != GS_F32) {
    using Tag = typename std::conditional<DT == GS_BF16, BF16Tag, F16Tag>::type;
    const uint16_t* xs = reinterpret_cast<const uint16_t*>(x);
    // vector body needs x 16-byte and q 8-byte aligned at the same element
    int64_t head = (int64_t)(((16u - ((uint32_t)(uintptr_t)xs & 15u)) & 15u) >> 1);
    if (head > n) head = n;
    if ((((uintptr_t)(q + head)) & 7u) != 0) head = n;
    for (int64_t i = tid; i < head; i += nthreads) q[i] = quant_one<FMT>(load_f<DT>(x, i), s, r, fin);
    const int64_t nv = (n - head) >> 3;
    const uint4* x8 = reinterpret_cast<const uint4*>(xs + head);
    uint2* q8 = reinterpret_cast<uint2*>(q + head);
    const int64_t n_it = (nv + kPass2It - 1) / kPass2It;
    for (int64_t run = blockIdx.x; run * kPass2Run < n_it; run += gridDim.x) {
      for (int k = 0; k < kPass2Run; ++k) {
        const int64_t from_end = run * kPass2Run + k;
        if (from_end >= n_it) break;
        const int64_t v0 = (n_it - 1 - from_end) * kPass2It + threadIdx.x;
        if (v0 + 3 * kQuantThreads < nv) {
          uint4 a[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) a[u] = ld_stream(x8 + v0 + u * kQuantThreads);
          uint32_t in[16], c[8];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            in[4 * u] = a[u].x;
            in[4 * u + 1] = a[u].y;
            in[4 * u + 2] = a[u].z;
            in[4 * u + 3] = a[u].w;
          }
          quant_words<Tag, FMT, 16>(in, c, s, r);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            st_stream(q8 + v0 + u * kQuantThreads, make_uint2(c[2 * u], c[2 * u + 1]));
        } else {  // the last, partial iteration of the body
          for (int u = 0; u < 4; ++u) {
            const int64_t v = v0 + u * kQuantThreads;
            if (v >= nv) break;
            const uint4 a = ld_stream(x8 + v);
            const uint32_t in[4] = {a.x, a.y, a.z, a.w};
            uint32_t c[2];
            quant_words<Tag, FMT, 4>(in, c, s, r);
            st_stream(q8 + v, make_uint2(c[0], c[1]));
          }
        }
      }
    }
    for (int64_t i = head + nv * 8 + tid; i < n; i += nthreads)
      q[i] = quant_one<FMT>(load_f<DT>(x, i), s, r, fin);
  } else {
    // 16-byte vectors of four fp32 -> four codes (one 4-byte store) where x
    // is 16-byte and q 4-byte aligned at the same element
    const uint32_t* xs = reinterpret_cast<const uint32_t*>(x);
    int64_t head = (int64_t)(((16u - ((uint32_t)(uintptr_t)xs & 15u)) & 15u) >> 2);
    if (head > n) head = n;
    if ((((uintptr_t)(q + head)) & 3u) != 0) head = n;
    for (int64_t i = tid; i < head; i += nthreads) q[i] = quant_one<FMT>(load_f<DT>(x, i), s, r, fin);
    const int64_t nv = (n - head) >> 2;
    const uint4* x4 = reinterpret_cast<const uint4*>(xs + head);
    uint32_t* q4 = reinterpret_cast<uint32_t*>(q + head);
    const int64_t n_it = (nv + kPass2It - 1) / kPass2It;
    for (int64_t run = blockIdx.x; run * kPass2Run < n_it; run += gridDim.x) {
      for (int k = 0; k < kPass2Run; ++k) {
        const int64_t from_end = run * kPass2Run + k;
        if (from_end >= n_it) break;
        const int64_t v0 = (n_it - 1 - from_end) * kPass2It + threadIdx.x;
        if (v0 + 3 * kQuantThreads < nv) {
          uint4 a[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) a[u] = ld_stream(x4 + v0 + u * kQuantThreads);
          uint32_t in[16], c[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            in[4 * u] = a[u].x;
            in[4 * u + 1] = a[u].y;
            in[4 * u + 2] = a[u].z;
            in[4 * u + 3] = a[u].w;
          }
          quant_words_f32<FMT, 16>(in, c, s, r);
#pragma unroll
          for (int u = 0; u < 4; ++u) q4[v0 + u * kQuantThreads] = c[u];
        } else {  // the last, partial iteration of the body
          for (int u = 0; u < 4; ++u) {
            const int64_t v = v0 + u * kQuantThreads;
            if (v >= nv) break;
            const uint4 a = ld_stream(x4 + v);
            const uint32_t in[4] = {a.x, a.y, a.z, a.w};
            uint32_t c[1];
            quant_words_f32<FMT, 4>(in, c, s, r);
            q4[v] = c[0];
          }
        }
      }
    }
    for (int64_t i = head + nv * 4 + tid; i < n; i += nthreads)
      q[i] = quant_one<FMT>(load_f<DT>(x, i), s, r, fin);
  }
}

// ---- launch helpers ---------------------------------------------------------
template <typename K>
static int64_t persistent_grid(K kernel, int64_t work_items_per_cta_slot, int64_t n_items) {
  int occ = 0;
  if (kernel_blocks_per_sm((const void*)kernel, kQuantThreads, 0, &occ) != cudaSuccess) occ = 1;
  if (occ < 1) occ = 1;
  int64_t grid = (int64_t)sm_count() * occ;
  const int64_t need = (n_items + work_items_per_cta_slot - 1) / work_items_per_cta_slot;
  if (grid > need) grid = need;
  return grid < 1 ? 1 : grid;
}

template <int DT, int FMT>
static cudaError_t quant_1x128_t(const void* x, int64_t R, int64_t C, uint8_t* q, float* scales,
                                 cudaStream_t st) {
  const int64_t n_tiles = R * (C / 128);
  const uintptr_t xa = (uintptr_t)x, qa = (uintptr_t)q;
  if constexpr (DT != GS_F32) {
    if ((xa & 31u) == 0 && (qa & 31u) == 0) {
      using Tag = typename std::conditional<DT == GS_BF16, BF16Tag, F16Tag>::type;
      auto k = quant_1x128_v8x2<Tag, FMT>;
      // oversubscribed grid: 64 CTAs per SM (several waves; CTAs started late
      // even out the SMs -- measured best of 16 to 128), each pass of a CTA
      // moves 64 tiles
      int64_t grid = (int64_t)sm_count() * 64;
      const int64_t need = (n_tiles + 8 * (kQuantThreads / 32) - 1) / (8 * (kQuantThreads / 32));
      if (grid > need) grid = need;
      if (grid < 1) grid = 1;
      k<<<(unsigned)grid, kQuantThreads, 0, st>>>(reinterpret_cast<const uint8_t*>(x), n_tiles, q,
                                                  scales);
      return cudaGetLastError();
    }
    if ((xa & 31u) == 0 && (qa & 15u) == 0) {
      using Tag = typename std::conditional<DT == GS_BF16, BF16Tag, F16Tag>::type;
      auto k = quant_1x128_v8<Tag, FMT>;
      // oversubscribed grid: 16 CTAs per SM, each pass of a CTA moves 64 tiles
      int64_t grid = (int64_t)sm_count() * 16;
      const int64_t need = (n_tiles + 4 * (kQuantThreads / 32) * kQ8Unroll - 1) /
                           (4 * (kQuantThreads / 32) * kQ8Unroll);
      if (grid > need) grid = need;
      if (grid < 1) grid = 1;
      k<<<(unsigned)grid, kQuantThreads, 0, st>>>(reinterpret_cast<const uint8_t*>(x), n_tiles, q,
                                                  scales);
      return cudaGetLastError();
    }
    if ((xa & 15u) == 0 && (qa & 7u) == 0) {
      using Tag = typename std::conditional<DT == GS_BF16, BF16Tag, F16Tag>::type;
      auto k = quant_1x128_v16<Tag, FMT>;
      // 16 tiles (8 warps x 2) per CTA per unrolled slot
      const int64_t grid = persistent_grid(k, (kQuantThreads / 16) * kQuantUnroll, n_tiles);
      k<<<(unsigned)grid, kQuantThreads, 0, st>>>(reinterpret_cast<const uint4*>(x), n_tiles,
                                                   reinterpret_cast<uint2*>(q), scales);
      return cudaGetLastError();
    }
  } else {
    if ((xa & 31u) == 0 && (qa & 15u) == 0) {
      auto k = quant_1x128_f32_v8<FMT>;
      // 64 CTAs per SM, several waves, as for the 16-bit kernel; each pass of
      // a CTA moves 32 tiles
      int64_t grid = (int64_t)sm_count() * 64;
      const int64_t need = (n_tiles + 4 * (kQuantThreads / 32) - 1) / (4 * (kQuantThreads / 32));
      if (grid > need) grid = need;
      if (grid < 1) grid = 1;
      k<<<(unsigned)grid, kQuantThreads, 0, st>>>(reinterpret_cast<const uint8_t*>(x), n_tiles, q,
                                                  scales);
      return cudaGetLastError();
    }
    if ((xa & 15u) == 0 && (qa & 3u) == 0) {
      auto k = quant_1x128_v32<FMT>;
      const int64_t grid = persistent_grid(k, kQuantThreads / 32, n_tiles);
      k<<<(unsigned)grid, kQuantThreads, 0, st>>>(reinterpret_cast<const uint4*>(x), n_tiles,
                                                  reinterpret_cast<uint32_t*>(q), scales);
      return cudaGetLastError();
    }
  }
  auto k = quant_1x128_any<DT, FMT>;
  const int64_t grid = persistent_grid(k, kQuantThreads / 32, n_tiles);
  k<<<(unsigned)grid, kQuantThreads, 0, st>>>(x, n_tiles, q, scales);
  return cudaGetLastError();
}

template <int FMT>
static cudaError_t quant_1x128_f(const void* x, int dt, int64_t R, int64_t C, uint8_t* q,
                                 float* scales, cudaStream_t st) {
  if (dt == GS_BF16) return quant_1x128_t<GS_BF16, FMT>(x, R, C, q, scales, st);
  if (dt == GS_F16) return quant_1x128_t<GS_F16, FMT>(x, R, C, q, scales, st);
  return quant_1x128_t<GS_F32, FMT>(x, R, C, q, scales, st);
}

cudaError_t launch_quant_1x128(const void* x, int dtype, int64_t R, int64_t C, int fmt, uint8_t* q,
                               float* scales, cudaStream_t stream) {
  if (R == 0 || C == 0) return cudaSuccess;
  return fmt == GS_E4M3 ? quant_1x128_f<GS_E4M3>(x, dtype, R, C, q, scales, stream)
                        : quant_1x128_f<GS_E5M2>(x, dtype, R, C, q, scales, stream);
}

template <int DT, int FMT>
cudaError_t quant_128x128_simple_t(const void* x, int64_t R, int64_t C, uint8_t* q, float* scales,
                                   cudaStream_t st) {
  auto k = quant_128x128_any<DT, FMT>;
  const int64_t grid = persistent_grid(k, 1, (R / 128) * (C / 128));
  k<<<(unsigned)grid, kQuantThreads, 0, st>>>(x, R, C, q, scales);
  return cudaGetLastError();
}

template <typename Tag, int FMT>
static cudaError_t quant_128x128_v8_t(const void* x, int64_t R, int64_t C, uint8_t* q,
                                      float* scales, cudaStream_t st) {
  auto k = quant_128x128_v8<Tag, FMT>;
  int occ = 0;
  const cudaError_t e = kernel_blocks_per_sm((const void*)k, kQ128Threads, 0, &occ);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  const int64_t nbr = R / 128, nbc = C / 128;
  int64_t grid = (int64_t)sm_count() * occ;
  if (grid > nbr * nbc) grid = nbr * nbc;
  k<<<(unsigned)grid, kQ128Threads, 0, st>>>(reinterpret_cast<const uint8_t*>(x), nbr, nbc, q, C,
                                             scales);
  return cudaGetLastError();
}

template <int FMT>
static cudaError_t quant_128x128_f32_v8_t(const void* x, int64_t R, int64_t C, uint8_t* q,
                                          float* scales, cudaStream_t st) {
  auto k = quant_128x128_f32_v8<FMT>;
  int occ = 0;
  const cudaError_t e = kernel_blocks_per_sm((const void*)k, kQ128Threads, 0, &occ);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  const int64_t nbr = R / 128, nbc = C / 128;
  int64_t grid = (int64_t)sm_count() * occ;
  if (grid > nbr * nbc) grid = nbr * nbc;
  k<<<(unsigned)grid, kQ128Threads, 0, st>>>(reinterpret_cast<const uint8_t*>(x), nbr, nbc, q, C,
                                             scales);
  return cudaGetLastError();
}

cudaError_t launch_quant_128x128_v8(const void* x, int dtype, int64_t R, int64_t C, int fmt,
                                    uint8_t* q, float* scales, cudaStream_t st) {
  if (R == 0 || C == 0) return cudaSuccess;
  if (dtype == GS_F32)
    return fmt == GS_E4M3 ? quant_128x128_f32_v8_t<GS_E4M3>(x, R, C, q, scales, st)
                          : quant_128x128_f32_v8_t<GS_E5M2>(x, R, C, q, scales, st);
  if (fmt == GS_E4M3)
    return dtype == GS_BF16 ? quant_128x128_v8_t<BF16Tag, GS_E4M3>(x, R, C, q, scales, st)
                            : quant_128x128_v8_t<F16Tag, GS_E4M3>(x, R, C, q, scales, st);
  return dtype == GS_BF16 ? quant_128x128_v8_t<BF16Tag, GS_E5M2>(x, R, C, q, scales, st)
                          : quant_128x128_v8_t<F16Tag, GS_E5M2>(x, R, C, q, scales, st);
}

cudaError_t launch_quant_128x128_simple(const void* x, int dtype, int64_t R, int64_t C, int fmt,
                                        uint8_t* q, float* scales, cudaStream_t st) {
  if (R == 0 || C == 0) return cudaSuccess;
  if (fmt == GS_E4M3) {
    if (dtype == GS_BF16) return quant_128x128_simple_t<GS_BF16, GS_E4M3>(x, R, C, q, scales, st);
    if (dtype == GS_F16) return quant_128x128_simple_t<GS_F16, GS_E4M3>(x, R, C, q, scales, st);
    return quant_128x128_simple_t<GS_F32, GS_E4M3>(x, R, C, q, scales, st);
  }
  if (dtype == GS_BF16) return quant_128x128_simple_t<GS_BF16, GS_E5M2>(x, R, C, q, scales, st);
  if (dtype == GS_F16) return quant_128x128_simple_t<GS_F16, GS_E5M2>(x, R, C, q, scales, st);
  return quant_128x128_simple_t<GS_F32, GS_E5M2>(x, R, C, q, scales, st);
}

template <typename Tag, int FMT>
static cudaError_t quant_128x128_v4_t(const void* x, int64_t R, int64_t C, uint8_t* q, float* scales,
                               cudaStream_t st) {
  auto k = quant_128x128_v4<Tag, FMT>;
  int occ = 0;
  const cudaError_t e = kernel_blocks_per_sm((const void*)k, kQ128Threads, 0, &occ);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  const int64_t nbr = R / 128, nbc = C / 128;
  int64_t grid = (int64_t)sm_count() * occ;
  if (grid > nbr * nbc) grid = nbr * nbc;
  k<<<(unsigned)grid, kQ128Threads, 0, st>>>(reinterpret_cast<const uint8_t*>(x), nbr, nbc, q, C,
                                             scales);
  return cudaGetLastError();
}

static cudaError_t launch_quant_128x128_v4(const void* x, int dtype, int64_t R, int64_t C, int fmt,
                                    uint8_t* q, float* scales, cudaStream_t st) {
  if (R == 0 || C == 0) return cudaSuccess;
  if (fmt == GS_E4M3)
    return dtype == GS_BF16 ? quant_128x128_v4_t<BF16Tag, GS_E4M3>(x, R, C, q, scales, st)
                            : quant_128x128_v4_t<F16Tag, GS_E4M3>(x, R, C, q, scales, st);
  return dtype == GS_BF16 ? quant_128x128_v4_t<BF16Tag, GS_E5M2>(x, R, C, q, scales, st)
                          : quant_128x128_v4_t<F16Tag, GS_E5M2>(x, R, C, q, scales, st);
}

cudaError_t launch_quant_128x128(const void* x, int dtype, int64_t R, int64_t C, int fmt,
                                 uint8_t* q, float* scales, cudaStream_t st) {
  if (R == 0 || C == 0) return cudaSuccess;
  const uintptr_t xa = (uintptr_t)x, qa = (uintptr_t)q;
  if ((xa & 31u) == 0 && (qa & (dtype == GS_F32 ? 7u : 15u)) == 0)
    return launch_quant_128x128_v8(x, dtype, R, C, fmt, q, scales, st);
  if (dtype != GS_F32 && (xa & 15u) == 0 && (qa & 7u) == 0)
    return launch_quant_128x128_v4(x, dtype, R, C, fmt, q, scales, st);
  return launch_quant_128x128_simple(x, dtype, R, C, fmt, q, scales, st);
}

template <int DT, int FMT>
static cudaError_t quant_tensor_t(const void* x, int64_t n, uint8_t* q, float* scale,
                                  uint32_t* partials, cudaStream_t st) {
  auto k1 = amax_partials<DT>;
  auto k2 = quant_tensor_pass2<DT, FMT>;
  int64_t g1 = persistent_grid(k1, kQuantThreads * 8, n);
  if (g1 > kMaxAmaxBlocks) g1 = kMaxAmaxBlocks;
  k1<<<(unsigned)g1, kQuantThreads, 0, st>>>(x, n, partials);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // pass 2: one CTA per run of kPass2Run iterations (many waves, highest
  // addresses first), at most 128 CTAs per SM so that the partials' reduction
  // at the start of every CTA stays small beside its data; the scalar head
  // and tail take one thread per element
  const int64_t vec = DT == GS_F32 ? 4 : 8;
  const int64_t runs = ((n / vec + kPass2It - 1) / kPass2It + kPass2Run - 1) / kPass2Run;
  int64_t g2 = runs;
  if (g2 > (int64_t)sm_count() * 128) g2 = (int64_t)sm_count() * 128;
  if (g2 < 1) g2 = 1;  // an empty tensor still gets its scale written
  k2<<<(unsigned)g2, kQuantThreads, 0, st>>>(x, n, q, scale, partials, (int)g1);
  return cudaGetLastError();
}

cudaError_t launch_quant_tensor(const void* x, int dtype, int64_t n, int fmt, uint8_t* q,
                                float* scale, uint32_t* partials, cudaStream_t st) {
  if (fmt == GS_E4M3) {
    if (dtype == GS_BF16) return quant_tensor_t<GS_BF16, GS_E4M3>(x, n, q, scale, partials, st);
    if (dtype == GS_F16) return quant_tensor_t<GS_F16, GS_E4M3>(x, n, q, scale, partials, st);
    return quant_tensor_t<GS_F32, GS_E4M3>(x, n, q, scale, partials, st);
  }
  if (dtype == GS_BF16) return quant_tensor_t<GS_BF16, GS_E5M2>(x, n, q, scale, partials, st);
  if (dtype == GS_F16) return quant_tensor_t<GS_F16, GS_E5M2>(x, n, q, scale, partials, st);
  return quant_tensor_t<GS_F32, GS_E5M2>(x, n, q, scale, partials, st);
}

}  // namespace gs
