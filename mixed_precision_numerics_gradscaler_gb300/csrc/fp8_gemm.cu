// fp8_gemm.cu -- the consumer of the block-scaled FP8 tiles: a GEMM on the
// 5th-generation tensor cores whose FP8 partial sums are promoted to FP32
// with their scales every 128 elements of K ("Loss scaling, FP8, and the
// failure that never crashes", section "FP8 needs a finer-grained fix than a
// single scale factor": periodic promotion to FP32 accumulation; "Mixed
// precision and FP8 training", section "FP8 training": promotion every 128
// elements, activations with 1x128 scales, weights with 128x128 scales).
//
//   D[m][n] = sum_kb sa[m][kb] * sb[n/128][kb] * sum_{k in kb} A[m][k] * B[n][k]
//
// A = [M, K] and B = [N, K] FP8 codes (both K-major, as fp8_quant_block
// writes them; each operand E4M3 or E5M2, the tensor cores take mixed
// pairs), D = [M, N] fp32 or bf16.  Persistent CTAs (one per SM) walk
// 128 x 256 tiles of D in groups of kGroupM tile rows (so the A and B panels
// in use at once stay in L2).  Each CTA has three warpgroups; setmaxnreg
// moves registers from the first (40 each) to the other two (232 each):
//   warp 0 (one lane)  TMA loads of the 128 x 128-byte A tile and the
//                      256 x 128-byte B tile of each K-block (128-byte
//                      swizzle, no multicast) into a 4-stage ring;
//   warp 1             allocates all 512 TMEM columns; one lane issues, per
//                      128-wide K-block, four tcgen05.mma.kind::f8f6f4
//                      (M 128, N 256, K 32) into one of two TMEM
//                      accumulators, then commits to the stage's "empty"
//                      barrier and the accumulator's "full" barrier;
//   warps 2-3          idle (they complete the first warpgroup);
//   warps 4-11         each reads one 32-row x 128-column quarter of the
//                      block's fp32 partial from TMEM (tcgen05.ld: warp w
//                      sees TMEM lanes 32 (w % 4) ...), multiplies by
//                      sa * sb and adds into fp32 registers (packed fp32x2
//                      fma: the promotion), releasing the accumulator as
//                      soon as its last TMEM read completes; after the
//                      tile's last K-block it stages its 32 x 128 piece of
//                      D in shared memory and writes it with TMA stores
//                      while the tensor cores already work on the next tile.
// Every wait is bounded by %globaltimer: a role that gives up records
// GS_ERR_TIMEOUT, raises a shared abort flag so the others leave their
// loops, waits (bounded) for its own loads or MMAs in flight, and the TMEM
// columns are freed on every path.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "gs_device.cuh"
#include "gs_internal.h"

namespace gs {

constexpr int kGB = 128;                   // tile M, K-block, weight block
constexpr int kGBN = 256;                  // tile N
constexpr int kGStages = 4;
constexpr int kGEpiWarps = 8;                    // warpgroups 1 and 2
constexpr int kGThreads = 128 + 32 * kGEpiWarps;  // warpgroup 0: TMA, MMA, 2 idle
// Register split (setmaxnreg): the CTA is launched with kGLaunchRegs per
// thread (65536 / 384 rounded down to a multiple of 8); warpgroup 0 gives
// back to kGCtrlRegs, warpgroups 1-2 grow to kGEpiRegs.  The shares must add
// up to the launch total exactly or the growing warps would wait forever.
constexpr int kGLaunchRegs = 168;
constexpr int kGCtrlRegs = 40;
constexpr int kGEpiRegs = 232;
static_assert(4 * kGCtrlRegs + kGEpiWarps * kGEpiRegs <= (kGThreads / 32) * kGLaunchRegs,
              "register split exceeds the launch allocation");
static_assert(kGThreads * kGLaunchRegs <= 65536, "launch allocation exceeds the register file");
constexpr int kGTileA = kGB * kGB;         // bytes of one A stage
constexpr int kGTileB = kGBN * kGB;        // bytes of one B stage
constexpr int kGStageBytes = kGTileA + kGTileB;
constexpr int kGTmemCols = 2 * kGBN;       // two 256-column fp32 accumulators
constexpr int kGOutBytes = 32 * 128;      // per promotion warp: 32 rows x 128 bytes of D
constexpr int kGSmemBytes = kGStages * kGStageBytes + kGEpiWarps * kGOutBytes + 1024 + 256;
static_assert(kGSmemBytes <= 232448, "dynamic shared memory above the per-CTA limit");
// Tile rows per raster group: B is read from DRAM once per group.  Measured
// on GB300 (16384 x 28672 x 8192): 16 rows read 2.02 GB per launch, 32 rows
// 1.19 GB at the same or a slightly higher rate, 40, 48 and 64 rows 1.64,
// 2.03 and 3.55 GB (the A panel of a group stops fitting in L2).
constexpr int kGroupM = 32;
constexpr uint64_t kGWaitNs = 2000000000ull;

__device__ __forceinline__ uint32_t g_smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t g_now() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool g_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(g_smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; gives up on timeout (setting the abort flag and the status)
// or when another role has already aborted.
__device__ __forceinline__ bool g_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                       int32_t* status) {
  if (g_try_wait(bar, parity)) return true;
  const uint64_t t0 = g_now();
  while (!g_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (g_now() - t0 > kGWaitNs) {
      *abort_flag = 1;
      atomicExch(status, (int32_t)GS_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}
// Bounded wait that ignores the abort flag (draining own work in flight).
__device__ __forceinline__ void g_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = g_now();
  while (!g_try_wait(bar, parity))
    if (g_now() - t0 > kGWaitNs) return;
}
__device__ __forceinline__ void g_bar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(g_smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void g_bar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(g_smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void g_tma_load(const CUtensorMap* map, uint64_t* bar, void* dst,
                                           int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(g_smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(g_smem_u32(bar))
      : "memory");
}
// TMA tile store from this CTA's shared memory (bulk-group completion).
__device__ __forceinline__ void g_tma_store(const CUtensorMap* map, const void* src, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map),
      "r"(x), "r"(y), "r"(g_smem_u32(src))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile in the 128-byte
// swizzled layout that TMA writes: rows of 128 bytes, 8-row groups 1024
// bytes apart (stride byte offset), descriptor version 1, swizzle mode
// 128B.  The leading byte offset is unused for swizzled K-major tiles.
__device__ __forceinline__ uint64_t umma_desc_k_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f8f6f4: fp32 accumulator, A and B each
// of its own FP8 format (0 E4M3, 1 E5M2), both K-major, N = 256, M = 128.
__host__ __device__ constexpr uint32_t umma_idesc_f8(uint32_t fmt_a, uint32_t fmt_b) {
  return (1u << 4) | (fmt_a << 7) | (fmt_b << 10) | ((uint32_t)(kGBN >> 3) << 17) |
         ((uint32_t)(kGB >> 4) << 24);
}

__device__ __forceinline__ void umma_f8(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          g_smem_u32(bar))
      : "memory");
}

// 32 lanes x 32 consecutive fp32 columns of TMEM -> 32 registers per thread
// (asynchronous: the registers may be read only after tmem_wait_ld).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// Waits for every tcgen05.ld of this thread; the registers of both loads are
// passed through so that nothing reads them before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&a)[32], uint32_t (&b)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]),
        "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]),
        "+r"(a[14]), "+r"(a[15]), "+r"(a[16]), "+r"(a[17]), "+r"(a[18]), "+r"(a[19]),
        "+r"(a[20]), "+r"(a[21]), "+r"(a[22]), "+r"(a[23]), "+r"(a[24]), "+r"(a[25]),
        "+r"(a[26]), "+r"(a[27]), "+r"(a[28]), "+r"(a[29]), "+r"(a[30]), "+r"(a[31]),
        "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]),
        "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]),
        "+r"(b[14]), "+r"(b[15]), "+r"(b[16]), "+r"(b[17]), "+r"(b[18]), "+r"(b[19]),
        "+r"(b[20]), "+r"(b[21]), "+r"(b[22]), "+r"(b[23]), "+r"(b[24]), "+r"(b[25]),
        "+r"(b[26]), "+r"(b[27]), "+r"(b[28]), "+r"(b[29]), "+r"(b[30]), "+r"(b[31])
      :
      : "memory");
}

// Two fp32 lanes in one 64-bit register, for the packed fused multiply-add
// (each lane is an IEEE fp32 fma, round to nearest even).
__device__ __forceinline__ uint64_t f32x2_pack(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_fma(uint64_t& acc, uint64_t v, uint64_t s) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(v), "l"(s));
}
__device__ __forceinline__ void f32x2_unpack(uint64_t p, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(p));
}

// Tile t of the raster -> (tile row, tile column), kGroupM tile rows at a
// time so that consecutive tiles share A and B panels.
__device__ __forceinline__ void gemm_tile_coords(int t, int tiles_m, int tiles_n, int& mt,
                                                 int& nt) {
  const int per_group = kGroupM * tiles_n;
  const int first_m = (t / per_group) * kGroupM;
  const int rows = min(kGroupM, tiles_m - first_m);
  const int r = t % per_group;
  mt = first_m + r % rows;
  nt = r / rows;
}

template <int FA, int FB, int OUT, bool TMA_STORE>
__global__ void __launch_bounds__(kGThreads, 1)
    gemm_fp8_block_scaled(const __grid_constant__ CUtensorMap map_a,
                          const __grid_constant__ CUtensorMap map_b,
                          const __grid_constant__ CUtensorMap map_d, const float* __restrict__ sa,
                          const float* __restrict__ sb, int64_t M, int64_t N, int64_t K,
                          void* __restrict__ d, int32_t* status, int stall) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment of the swizzled tiles
  const uint32_t pad = (1024u - (g_smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* tiles = smem_raw + pad;
  uint8_t* out_stage = tiles + kGStages * kGStageBytes;  // 1024-byte aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(out_stage + kGEpiWarps * kGOutBytes);
  uint64_t* empty = full + kGStages;
  uint64_t* tfull = empty + kGStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = (int)(K / kGB);
  const int tiles_m = (int)((M + kGB - 1) / kGB), tiles_n = (int)((N + kGBN - 1) / kGBN);
  const int n_tiles = tiles_m * tiles_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      g_bar_init(&full[s], 1);
      g_bar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      g_bar_init(&tfull[b], 1);
      g_bar_init(&tempty[b], 32 * kGEpiWarps);
    }
    g_bar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     g_smem_u32(tmem_slot)),
                 "r"(kGTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {  // warpgroup 0
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kGCtrlRegs));
    if (warp == 0 && lane == 0) {  // TMA producer
      uint32_t it = 0;  // K-blocks issued so far over this CTA's tiles (mod 2^32)
      bool go = !stall;  // stall: test hook, no loads, so the MMA's wait runs out
      for (int t = blockIdx.x; go && t < n_tiles; t += gridDim.x) {
        int mt, nt;
        gemm_tile_coords(t, tiles_m, tiles_n, mt, nt);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const uint32_t s = it % kGStages, ph = (it / kGStages) & 1u;
          if (!g_wait(&empty[s], ph ^ 1u, abort_flag, status)) {
            go = false;
            break;
          }
          uint8_t* st = tiles + s * kGStageBytes;
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                           g_smem_u32(&full[s])),
                       "r"(kGStageBytes)
                       : "memory");
          g_tma_load(&map_a, &full[s], st, kb * kGB, mt * kGB);
          g_tma_load(&map_b, &full[s], st + kGTileA, kb * kGB, nt * kGBN);
        }
      }
      // Let the last load of every stage land before the CTA can exit (they
      // have landed already unless another role gave up).
      const uint32_t issued_tail = it < kGStages ? it : kGStages;
      for (uint32_t j = it - issued_tail; j != it; ++j)
        g_drain(&full[j % kGStages], (j / kGStages) & 1u);
    } else if (warp == 1 && lane == 0) {  // MMA issuer
      constexpr uint32_t idesc = umma_idesc_f8((uint32_t)FA, (uint32_t)FB);
      uint32_t it = 0;
      bool go = true;
      for (int t = blockIdx.x; go && t < n_tiles; t += gridDim.x) {
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const uint32_t s = it % kGStages, b = it & 1u;
          const uint32_t ph = (it / kGStages) & 1u, tph = (it >> 1) & 1u;
          if (!g_wait(&full[s], ph, abort_flag, status) ||
              !g_wait(&tempty[b], tph ^ 1u, abort_flag, status)) {
            go = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = g_smem_u32(tiles + s * kGStageBytes);
          const uint32_t b0 = a0 + kGTileA;
#pragma unroll
          for (int kk = 0; kk < kGB / 32; ++kk)
            umma_f8(tmem + b * kGBN, umma_desc_k_sw128(a0 + 32 * kk),
                    umma_desc_k_sw128(b0 + 32 * kk), idesc, kk > 0 ? 1u : 0u);
          umma_commit(&empty[s]);
          umma_commit(&tfull[b]);
        }
      }
      umma_commit(drain);  // completes when every MMA issued above has
      g_drain(drain, 0);
    }
  } else {  // promotion and store: warpgroups 1 and 2
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kGEpiRegs));
    const int q = warp & 3;               // TMEM lane quarter this warp may read
    const int h = (warp - 4) >> 2;        // which 128 columns of the 256
    const int row = 32 * q + lane;
    // Store this thread's 128 promoted values of row m, columns n0.. of D.
    // TMA path (all 32 lanes call it): each 128-byte column chunk of the
    // warp's 32 rows is written to its staging buffer in the 128-byte
    // swizzled layout (16-byte piece p of row r at p ^ (r % 8)) and stored
    // by one TMA instruction, which also clips rows and columns past D.
    uint8_t* const my_out = out_stage + (warp - 4) * kGOutBytes;
    // `between` runs once the first chunk is handed to TMA, overlapping the
    // wait for its buffer (or before the element stores).
    auto store_tile = [&](int64_t m, int64_t n0, bool live, const uint64_t (&acc)[kGB / 2],
                          auto&& between) {
      if constexpr (TMA_STORE) {
        if (!__any_sync(0xffffffffu, live)) {
          between();
          return;
        }
        constexpr int kCols = OUT == GS_F32 ? 32 : 64;  // columns per 128-byte chunk
#pragma unroll
        for (int c = 0; c < kGB / kCols; ++c) {
          if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          __syncwarp();  // the previous chunk has been read out of the buffer
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            float o[8];  // this 16-byte piece's values (4 fp32 or 8 bf16)
#pragma unroll
            for (int j = 0; j < (OUT == GS_F32 ? 2 : 4); ++j)
              f32x2_unpack(acc[c * kCols / 2 + (OUT == GS_F32 ? 2 : 4) * p + j], o[2 * j],
                           o[2 * j + 1]);
            uint4 v;
            if constexpr (OUT == GS_F32)
              v = make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                             __float_as_uint(o[3]));
            else
              v = make_uint4(cvt_f32x2_bf16x2(o[1], o[0]), cvt_f32x2_bf16x2(o[3], o[2]),
                             cvt_f32x2_bf16x2(o[5], o[4]), cvt_f32x2_bf16x2(o[7], o[6]));
            *reinterpret_cast<uint4*>(my_out + lane * 128 + ((p ^ (lane & 7)) << 4)) = v;
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            g_tma_store(&map_d, my_out, (int32_t)(n0 + c * kCols), (int32_t)(m - lane));
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          }
          if (c == 0) between();
        }
      } else {  // unaligned D or row stride: one element at a time
        between();
        if (!live) return;
        const int64_t off = m * N + n0;
#pragma unroll
        for (int j = 0; j < kGB / 2; ++j) {
          float lo, hi;
          f32x2_unpack(acc[j], lo, hi);
          if constexpr (OUT == GS_F32) {
            if (n0 + 2 * j < N) reinterpret_cast<float*>(d)[off + 2 * j] = lo;
            if (n0 + 2 * j + 1 < N) reinterpret_cast<float*>(d)[off + 2 * j + 1] = hi;
          } else {
            const uint32_t pr = cvt_f32x2_bf16x2(hi, lo);
            if (n0 + 2 * j < N) reinterpret_cast<uint16_t*>(d)[off + 2 * j] = (uint16_t)(pr & 0xFFFFu);
            if (n0 + 2 * j + 1 < N) reinterpret_cast<uint16_t*>(d)[off + 2 * j + 1] = (uint16_t)(pr >> 16);
          }
        }
      }
    };
    // Tile t's raster coordinates (mt = -1 past the last tile), and from
    // them this thread's row, column block and scale rows.
    auto coords = [&](int t, int& mt, int& nt) {
      mt = -1;
      nt = 0;
      if (t < n_tiles) gemm_tile_coords(t, tiles_m, tiles_n, mt, nt);
    };
    auto derive = [&](int mt, int nt, int64_t& m, int64_t& n0, bool& live, const float*& sa_row,
                      const float*& sb_row) {
      m = (int64_t)mt * kGB + row;
      n0 = (int64_t)nt * kGBN + h * kGB;
      live = mt >= 0 && m < M && n0 < N;  // rows / columns past the edge were zeros
      sa_row = sa + (live ? m * nkb : 0);
      sb_row = sb + (live ? (n0 / kGB) * nkb : 0);
    };
    int mt, nt, mt_n, nt_n;  // this tile and the next
    coords(blockIdx.x, mt, nt);
    coords(blockIdx.x + gridDim.x, mt_n, nt_n);
    int64_t m, n0;
    bool live;
    const float *sa_row, *sb_row;
    derive(mt, nt, m, n0, live, sa_row, sb_row);
    float sa_v = live ? sa_row[0] : 0.0f, sb_v = live ? sb_row[0] : 0.0f;
    const int kb_ahead = nkb > 4 ? nkb - 4 : 0;  // when to fetch the next tile's first scales
    uint32_t it = 0;
    bool go = true;
    for (int t = blockIdx.x; go && t < n_tiles; t += gridDim.x) {
      float sa_first_n = 0.0f, sb_first_n = 0.0f;
      uint64_t acc[kGB / 2];  // column pairs (2j, 2j + 1)
#pragma unroll
      for (int j = 0; j < kGB / 2; ++j) acc[j] = 0ull;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const uint32_t b = it & 1u;
        const float sc = __fmul_rn(sa_v, sb_v);
        const uint64_t sc2 = f32x2_pack(__float_as_uint(sc), __float_as_uint(sc));
        if (live && kb + 1 < nkb) {  // next block's scales, ahead of the wait
          sa_v = sa_row[kb + 1];
          sb_v = sb_row[kb + 1];
        }
        if (kb == kb_ahead) {  // the next tile's, well ahead of its start
          int64_t m_x, n0_x;
          bool live_x;
          const float *sa_x, *sb_x;
          derive(mt_n, nt_n, m_x, n0_x, live_x, sa_x, sb_x);
          if (live_x) {
            sa_first_n = sa_x[0];
            sb_first_n = sb_x[0];
          }
        }
        // the warp leaves together: tcgen05.ld below needs all 32 lanes
        const bool got = g_wait(&tfull[b], (it >> 1) & 1u, abort_flag, status);
        if (!__all_sync(0xffffffffu, got)) {
          go = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + b * kGBN + h * kGB;
        uint32_t v0[32], v1[32];  // 64 columns per wait
        tmem_ld32(taddr, v0);
        tmem_ld32(taddr + 32, v1);
        tmem_wait_ld(v0, v1);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          f32x2_fma(acc[j], f32x2_pack(v0[2 * j], v0[2 * j + 1]), sc2);
          f32x2_fma(acc[16 + j], f32x2_pack(v1[2 * j], v1[2 * j + 1]), sc2);
        }
        tmem_ld32(taddr + 64, v0);
        tmem_ld32(taddr + 96, v1);
        tmem_wait_ld(v0, v1);
        // Every TMEM read of this block is done: hand the accumulator back
        // to the MMA before the last FMAs.
        tc_fence_before();
        g_bar_arrive(&tempty[b]);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          f32x2_fma(acc[32 + j], f32x2_pack(v0[2 * j], v0[2 * j + 1]), sc2);
          f32x2_fma(acc[48 + j], f32x2_pack(v1[2 * j], v1[2 * j + 1]), sc2);
        }
      }
      if (!go || *abort_flag) break;
      int mt_2, nt_2;  // the tile after next, located while TMA drains
      store_tile(m, n0, live, acc, [&] { coords(t + 2 * (int)gridDim.x, mt_2, nt_2); });
      derive(mt_n, nt_n, m, n0, live, sa_row, sb_row);
      mt_n = mt_2;
      nt_n = nt_2;
      sa_v = sa_first_n;
      sb_v = sb_first_n;
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // D written
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kGTmemCols)
                 : "memory");
  }
}

static PFN_cuTensorMapEncodeTiled_v12000 gemm_encode_fn() {
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

static CUresult encode_k_major(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t K,
                               uint32_t box_rows) {
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K};
  const cuuint32_t box[2] = {kGB, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return gemm_encode_fn()(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int FA, int FB, int OUT, bool TMA_STORE>
static cudaError_t gemm_t(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& md,
                          const float* sa, const float* sb, int64_t M, int64_t N, int64_t K,
                          void* d, int32_t* status, cudaStream_t st) {
  auto k = gemm_fp8_block_scaled<FA, FB, OUT, TMA_STORE>;
  // The setmaxnreg split is sized for exactly kGLaunchRegs per thread at
  // launch; a build that allocated another count must not run.
  static std::once_flag once;
  static cudaError_t regs_err = cudaSuccess;
  std::call_once(once, [&] {
    cudaFuncAttributes fa;
    regs_err = cudaFuncGetAttributes(&fa, k);
    if (regs_err == cudaSuccess && fa.numRegs != kGLaunchRegs)
      regs_err = cudaErrorInvalidConfiguration;
  });
  if (regs_err != cudaSuccess) return regs_err;
  int occ = 0;  // also raises the shared-memory limit in this context
  const cudaError_t e = kernel_blocks_per_sm((const void*)k, kGThreads, kGSmemBytes, &occ);
  if (e != cudaSuccess) return e;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  const int64_t tiles = ((M + kGB - 1) / kGB) * ((N + kGBN - 1) / kGBN);
  const unsigned grid = (unsigned)std::min<int64_t>(tiles, (int64_t)sm_count());
  k<<<grid, kGThreads, kGSmemBytes, st>>>(ma, mb, md, sa, sb, M, N, K, d, status, test_stall());
  return cudaGetLastError();
}

template <int FA, int FB>
static cudaError_t gemm_fmt(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& md,
                            const float* sa, const float* sb, int64_t M, int64_t N, int64_t K,
                            bool f32, bool tma_store, void* d, int32_t* status, cudaStream_t st) {
  if (tma_store)
    return f32 ? gemm_t<FA, FB, GS_F32, true>(ma, mb, md, sa, sb, M, N, K, d, status, st)
               : gemm_t<FA, FB, GS_BF16, true>(ma, mb, md, sa, sb, M, N, K, d, status, st);
  return f32 ? gemm_t<FA, FB, GS_F32, false>(ma, mb, md, sa, sb, M, N, K, d, status, st)
             : gemm_t<FA, FB, GS_BF16, false>(ma, mb, md, sa, sb, M, N, K, d, status, st);
}

// The caller has checked: qa and qb 16-byte aligned, K a multiple of 128,
// M, N, K below 2^31 and fewer than 2^30 tiles.  Returns
// cudaErrorNotSupported when the tensor-map entry point is missing.
cudaError_t launch_gemm_fp8_block_scaled(const uint8_t* qa, const float* sa, const uint8_t* qb,
                                         const float* sb, int64_t M, int64_t N, int64_t K,
                                         int fmt_a, int fmt_b, int out_dtype, void* d,
                                         int32_t* status, cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  const size_t esz = out_dtype == GS_F32 ? 4 : 2;
  if (K == 0) return cudaMemsetAsync(d, 0, (size_t)M * (size_t)N * esz, st);  // empty sums
  if (!gemm_encode_fn()) return cudaErrorNotSupported;
  CUtensorMap ma, mb;
  if (encode_k_major(&ma, qa, M, K, kGB) != CUDA_SUCCESS ||
      encode_k_major(&mb, qb, N, K, kGBN) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // D through TMA stores when its base and row stride allow it (16 bytes).
  CUtensorMap md;
  memset(&md, 0, sizeof(md));
  int tma_store = ((uintptr_t)d % 16 == 0) && (((size_t)N * esz) % 16 == 0);
  if (tma_store) {
    const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)N * esz};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / esz), 32};
    const cuuint32_t estr[2] = {1, 1};
    if (gemm_encode_fn()(&md,
                         out_dtype == GS_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                             : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         2, d, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const bool f32 = out_dtype == GS_F32, tma = tma_store != 0;
  if (fmt_a == GS_E4M3)
    return fmt_b == GS_E4M3
               ? gemm_fmt<GS_E4M3, GS_E4M3>(ma, mb, md, sa, sb, M, N, K, f32, tma, d, status, st)
               : gemm_fmt<GS_E4M3, GS_E5M2>(ma, mb, md, sa, sb, M, N, K, f32, tma, d, status, st);
  return fmt_b == GS_E4M3
             ? gemm_fmt<GS_E5M2, GS_E4M3>(ma, mb, md, sa, sb, M, N, K, f32, tma, d, status, st)
             : gemm_fmt<GS_E5M2, GS_E5M2>(ma, mb, md, sa, sb, M, N, K, f32, tma, d, status, st);
}

}  // namespace gs
