// gs_internal.h -- host-side declarations shared by the library's
// translation units (kernel launchers, the chunk table, device queries).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "gs_layout.h"

namespace gs {

// Cached device properties of the current device.
int sm_count();

// Resident blocks per SM of `kernel` at (threads, dynamic smem bytes) in the
// CUDA context current on this thread; the first call per kernel and context
// also raises the kernel's dynamic shared-memory limit there (function
// attributes belong to the module loaded in a context, so a new primary
// context after cudaDeviceReset needs them again).  Thread-safe; cached
// under the context's ID.
cudaError_t kernel_blocks_per_sm(const void* kernel, int threads, int smem_bytes, int* blocks);
int current_device();

// ID of the CUDA context current on this thread (0 and true when none is
// current yet; false when the driver cannot be queried).  The driver never
// hands out an ID twice in a process, whereas a new context may reuse a
// destroyed one's handle, so caches of per-context state use the ID as key.
bool current_context_id(unsigned long long* id);

// Device address of the module global `symbol` (a __device__ variable of
// this library) in the CUDA context current on this thread.  Every context
// that loads the library holds its own copy of each global at its own
// address, so the address is looked up with cudaGetSymbolAddress on the
// first call in a context and cached under the context's ID (a fixed table,
// no heap allocation).  Thread-safe.
cudaError_t symbol_address(const void* symbol, void** out);

// Records e as the calling thread's last CUDA error (gs_last_cuda_error).
void record_cuda_error(cudaError_t e);
// True if the current device can dereference p as given: its own device
// memory, managed memory, or mapped host memory whose device address is p.
bool device_reachable(const void* p);

// A byte range [lo, hi) of memory.
struct Span {
  uintptr_t lo, hi;
};
// True when two written ranges overlap each other, or a written range
// overlaps a read one (empty ranges never do).  Sorts `writes` in place;
// O((writes + reads) log writes).
bool spans_conflict(Span* writes, size_t n_writes, const Span* reads, size_t n_reads);

// Test hook (gs_test_set_stall): nonzero makes the block-scaled FP8 GEMM issue
// no TMA loads, so that its bounded waits run out.
int test_stall();

// Launchers.  Each returns the launch's cudaError_t.
cudaError_t launch_unscale_check_update(const Chunk* d_chunks, int64_t n_chunks, ListWs* ws,
                                        float* scale, int32_t* tracker, int32_t* found,
                                        int64_t* skipped, float growth, float backoff,
                                        int32_t interval, cudaStream_t stream,
                                        ScalerPolicy policy = ScalerPolicy{nullptr, 1, 0, 0.0f},
                                        float* grad_norm = nullptr, double* norm_slots = nullptr);
cudaError_t launch_master_update_sgd(const MChunk* d_chunks, int64_t n_chunks, float lr,
                                     float max_norm, const float* grad_norm,
                                     const int32_t* found_inf, cudaStream_t stream);

cudaError_t launch_quant_1x128(const void* x, int dtype, int64_t R, int64_t C, int fmt, uint8_t* q,
                               float* scales, cudaStream_t stream);
cudaError_t launch_quant_128x128(const void* x, int dtype, int64_t R, int64_t C, int fmt,
                                 uint8_t* q, float* scales, cudaStream_t stream);
// The 128x128 kernels behind launch_quant_128x128: direct 32-byte loads
// (x 32-byte aligned; q 16-byte aligned for 16-bit input, 8-byte for FP32),
// direct 16-byte loads (16-bit x 16-byte aligned, q 8-byte aligned), and one
// CTA per block for any dtype and alignment.
cudaError_t launch_quant_128x128_v8(const void* x, int dtype, int64_t R, int64_t C, int fmt,
                                    uint8_t* q, float* scales, cudaStream_t stream);
cudaError_t launch_quant_128x128_simple(const void* x, int dtype, int64_t R, int64_t C, int fmt,
                                        uint8_t* q, float* scales, cudaStream_t stream);
cudaError_t launch_quant_tensor(const void* x, int dtype, int64_t n, int fmt, uint8_t* q,
                                float* scale, uint32_t* partials, cudaStream_t stream);
cudaError_t launch_dequant(const uint8_t* q, const float* scales, int64_t R, int64_t C,
                           int block_r, int block_c, int fmt, int out_dtype, void* y,
                           cudaStream_t stream);
cudaError_t launch_quant_mx(const void* x, int dtype, int64_t R, int64_t C, int fmt, uint8_t* q,
                            uint8_t* scales, cudaStream_t stream);
cudaError_t launch_dequant_mx(const uint8_t* q, const uint8_t* scales, int64_t R, int64_t C,
                              int fmt, int out_dtype, void* y, cudaStream_t stream);
cudaError_t launch_quant_tensor_delayed(const void* x, int dtype, int64_t n, int fmt, uint8_t* q,
                                        float* history, int hist_len, int32_t* pos,
                                        float* scale_used, uint32_t* partials, cudaStream_t stream);
cudaError_t launch_gemm_fp8_block_scaled(const uint8_t* qa, const float* sa, const uint8_t* qb,
                                         const float* sb, int64_t M, int64_t N, int64_t K,
                                         int fmt_a, int fmt_b, int out_dtype, void* d,
                                         int32_t* status, cudaStream_t stream);
cudaError_t launch_set_state(float* scale, int32_t* tracker, float h_scale, int32_t h_tracker,
                             cudaStream_t stream);

// Number of per-CTA amax partials the per-tensor path may write.
constexpr int kMaxAmaxBlocks = 2048;

}  // namespace gs
