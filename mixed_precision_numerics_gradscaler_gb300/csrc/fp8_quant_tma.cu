// fp8_quant_tma.cu -- 128x128 block-scaled FP8 quantisation of 16-bit
// weights with TMA staging ("Loss scaling, FP8, and the failure that never
// crashes", section "FP8 needs a finer-grained fix than a single scale
// factor", and "Mixed precision and FP8 training", section "FP8 training":
// one FP32 scale per 128x128 weight block).
//
// Inputs whose base is 32-byte aligned (with 16-byte aligned codes) go to
// the direct-load kernel quant_128x128_v8 in fp8_quant.cu, which measured
// faster; this kernel takes 16-byte aligned inputs, the alignment a TMA
// tensor map needs, and anything less goes to the one-CTA-per-block kernel.
//
// A persistent CTA walks its share of the blocks.  One elected thread
// issues cp.async.bulk.tensor.2d loads of whole 128x128 tiles (32 KB,
// no swizzle, no multicast) into a 3-stage ring, each stage guarded by an
// mbarrier with a transaction count.  All 512 threads then pull the tile
// from shared memory into registers (4 x 16 B each, conflict-free rows of
// 256 B), reduce the block amax (packed 16-bit max, warp shuffle, one word
// per warp), release the stage so the next load overlaps the cast, cast
// through quant_words (the packed f32x2 exact quotient) and write FP8 codes
// straight from registers with 8-byte coalesced stores.
// Every wait on an mbarrier is bounded by %globaltimer; a CTA that gives
// up records GS_ERR_TIMEOUT in the device status word, waits (bounded) for
// its own loads still in flight, and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "gs_device.cuh"
#include "gs_quant.cuh"
#include "gs_internal.h"

namespace gs {

constexpr int kTmaThreads = 512;
constexpr int kTmaWarps = kTmaThreads / 32;
constexpr int kRowsPerPass = kTmaThreads / 16;   // 16 threads cover a 256-byte row
constexpr int kRowPasses = 128 / kRowsPerPass;
constexpr int kTmaStages = 3;
constexpr int kTileBytes = 128 * 128 * 2;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
// tiles, then the stage barriers, then (16-byte aligned) two rows of
// per-warp maxima
constexpr int kRedOffset = (kTmaStages * kTileBytes + kTmaStages * 8 + 15) / 16 * 16;
constexpr int kTmaSmemBytes = kRedOffset + 2 * kTmaWarps * 4 + 64;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  return true;
}
__device__ __forceinline__ void tma_load_tile(const CUtensorMap* map, uint64_t* bar, void* dst,
                                              int32_t col, int32_t row) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(kTileBytes)
               : "memory");
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(col), "r"(row), "r"(smem_u32(bar))
      : "memory");
}

template <typename Tag, int FMT>
__global__ void __launch_bounds__(kTmaThreads)
    quant_128x128_tma(const __grid_constant__ CUtensorMap map, int64_t nbr, int64_t nbc,
                      uint8_t* __restrict__ q, int64_t C, float* __restrict__ scales,
                      int32_t* status, int stall) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* tiles = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTmaStages * kTileBytes);
  uint32_t* red = reinterpret_cast<uint32_t*>(smem + kRedOffset);  // [2][kTmaWarps]

  const int64_t n_blocks = nbr * nbc;
  if ((int64_t)blockIdx.x >= n_blocks) return;
  const int64_t my_n = (n_blocks - 1 - blockIdx.x) / gridDim.x + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kTmaStages; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // Block b = blockIdx.x + k * gridDim.x is (row b / nbc, column b % nbc);
  // walking k, both advance by gridDim.x's quotient and remainder, so no
  // division is left in the loop.
  const int64_t step_r = gridDim.x / nbc, step_c = gridDim.x % nbc;
  auto advance = [&](int64_t& br, int64_t& bc) {
    br += step_r;
    bc += step_c;
    if (bc >= nbc) {
      bc -= nbc;
      ++br;
    }
  };
  int64_t ibr = blockIdx.x / nbc, ibc = blockIdx.x % nbc;  // next block to load
  uint32_t istage = 0;
  int64_t issued = 0;
  auto issue = [&]() {
    tma_load_tile(&map, &full[istage], tiles + istage * kTileBytes, (int32_t)(ibc * 128),
                  (int32_t)(ibr * 128));
    advance(ibr, ibc);
    istage = istage + 1 == kTmaStages ? 0 : istage + 1;
    ++issued;
  };
  if (tid == 0 && !stall)  // stall: test hook, no loads, so the first wait runs out
    while (issued < kTmaStages && issued < my_n) issue();

  // Thread tid owns rows (tid >> 4) + kRowsPerPass * j, 16-byte column chunk
  // (tid & 15): a warp reads two whole 256-byte rows per pass.
  const int row0 = tid >> 4, chunk = tid & 15;
  int64_t br = blockIdx.x / nbc, bc = blockIdx.x % nbc;  // this block
  uint32_t stage = 0, phase = 0;
  for (int64_t k = 0; k < my_n; ++k) {
    const bool ok = mbar_wait_bounded(&full[stage], phase);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        atomicExch(status, (int32_t)GS_ERR_TIMEOUT);
        // let the loads of this CTA still in flight land before exiting
        for (int64_t j = k; j < issued; ++j)
          (void)mbar_wait_bounded(&full[j % kTmaStages], (uint32_t)((j / kTmaStages) & 1));
      }
      __syncthreads();
      return;
    }
    const uint4* tile = reinterpret_cast<const uint4*>(tiles + stage * kTileBytes);
    uint4 v[kRowPasses];
#pragma unroll
    for (int j = 0; j < kRowPasses; ++j) v[j] = tile[(row0 + kRowsPerPass * j) * 16 + chunk];
    const uint32_t mm = 0x7FFF7FFFu;
    uint32_t m2 = 0;
#pragma unroll
    for (int j = 0; j < kRowPasses; ++j)
      m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(v[j].x & mm, v[j].y & mm), __vmaxu2(v[j].z & mm, v[j].w & mm)));
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    uint32_t* rb = red + (k & 1) * kTmaWarps;
    if (lane == 0) rb[warp] = m;
    __syncthreads();  // every thread holds its part of the tile: the stage is free
    if (tid == 0 && issued < my_n && !stall) issue();
    {
      const uint4* r4 = reinterpret_cast<const uint4*>(rb);
      uint4 a = r4[0];
#pragma unroll
      for (int w = 1; w < kTmaWarps / 4; ++w) {
        const uint4 c = r4[w];
        a = make_uint4(max(a.x, c.x), max(a.y, c.y), max(a.z, c.z), max(a.w, c.w));
      }
      m = max(max(a.x, a.y), max(a.z, a.w));
    }
    const float s = block_scale<FMT>(mag16_to_float<Tag>(m));
    const float r = __frcp_rn(s);
    const int64_t r0 = br * 128, c0 = bc * 128;
    if (tid == 0) scales[br * nbc + bc] = s;
    uint32_t in[4 * kRowPasses], c[2 * kRowPasses];
#pragma unroll
    for (int j = 0; j < kRowPasses; ++j) {
      in[4 * j] = v[j].x;
      in[4 * j + 1] = v[j].y;
      in[4 * j + 2] = v[j].z;
      in[4 * j + 3] = v[j].w;
    }
    quant_words<Tag, FMT, 4 * kRowPasses>(in, c, s, r);
#pragma unroll
    for (int j = 0; j < kRowPasses; ++j)
      st_stream(reinterpret_cast<uint2*>(q + (r0 + row0 + kRowsPerPass * j) * C + c0 + chunk * 8),
                make_uint2(c[2 * j], c[2 * j + 1]));
    advance(br, bc);
    if (++stage == kTmaStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

template <typename Tag, int FMT>
static cudaError_t launch_tma_t(const CUtensorMap& map, int64_t R, int64_t C, uint8_t* q,
                                float* scales, int32_t* status, cudaStream_t st) {
  auto k = quant_128x128_tma<Tag, FMT>;
  int occ = 0;
  const cudaError_t e = kernel_blocks_per_sm((const void*)k, kTmaThreads, kTmaSmemBytes, &occ);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  const int64_t nbr = R / 128, nbc = C / 128;
  int64_t grid = (int64_t)sm_count() * occ;
  if (grid > nbr * nbc) grid = nbr * nbc;
  k<<<(unsigned)grid, kTmaThreads, kTmaSmemBytes, st>>>(map, nbr, nbc, q, C, scales, status,
                                                        test_stall());
  return cudaGetLastError();
}

cudaError_t launch_quant_128x128(const void* x, int dtype, int64_t R, int64_t C, int fmt,
                                 uint8_t* q, float* scales, int32_t* status, cudaStream_t st) {
  if (R == 0 || C == 0) return cudaSuccess;
  if (((uintptr_t)x & 31u) == 0 && ((uintptr_t)q & (dtype == GS_F32 ? 7u : 15u)) == 0)
    return launch_quant_128x128_v8(x, dtype, R, C, fmt, q, scales, st);
  const bool tma_ok = dtype != GS_F32 && ((uintptr_t)x & 15u) == 0 && ((uintptr_t)q & 7u) == 0 &&
                      R < (int64_t(1) << 31) && C < (int64_t(1) << 31) && encode_fn() != nullptr;
  if (!tma_ok) return launch_quant_128x128_simple(x, dtype, R, C, fmt, q, scales, st);
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)R};
  const cuuint64_t strides[1] = {(cuuint64_t)C * 2};
  const cuuint32_t box[2] = {128, 128};
  const cuuint32_t estr[2] = {1, 1};
  CUresult cr = encode_fn()(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(x), dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return launch_quant_128x128_simple(x, dtype, R, C, fmt, q, scales, st);
  if (fmt == GS_E4M3)
    return dtype == GS_BF16 ? launch_tma_t<BF16Tag, GS_E4M3>(map, R, C, q, scales, status, st)
                            : launch_tma_t<F16Tag, GS_E4M3>(map, R, C, q, scales, status, st);
  return dtype == GS_BF16 ? launch_tma_t<BF16Tag, GS_E5M2>(map, R, C, q, scales, status, st)
                          : launch_tma_t<F16Tag, GS_E5M2>(map, R, C, q, scales, status, st);
}

}  // namespace gs
