// gs_noalloc.cu -- gs_unscale_check_update_noalloc: the GradScaler step for
// callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not available or not
// allowed -- inside a custom allocator's own callbacks, in a process whose
// device memory is fully reserved up front by another runtime, or in a
// plugin that must not create allocations it cannot free.  Such a caller
// cannot use gs_tensor_list_create, which allocates the chunk table.
//
// This variant keeps the chunk table and the epilogue words in one
// file-scope device array of fixed size, so nothing is allocated per call
// or ever: every GPU that loads the library holds the array until the
// process exits.  The tensor table travels by value as a kernel parameter;
// a one-CTA kernel expands it into chunks inside the array and clears the
// epilogue words; then the same unscale/check/update kernel as
// gs_unscale_check_update runs on it.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <cmath>

#include "gs_internal.h"
#include "gsfp8.h"

namespace gs {

// Scratch layout: [ListWs (256 B)] [Chunk x kNoAllocMaxChunks].
constexpr int64_t kNoAllocMaxChunks = 32768;  // 268,435,456 elements
constexpr size_t kNoAllocWsBytes = 256;
constexpr size_t kNoAllocScratchBytes = kNoAllocWsBytes + kNoAllocMaxChunks * sizeof(Chunk);
constexpr int kNoAllocMaxTensors = 960;       // keeps the table under the kernel-parameter limit

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct TensorTable {
  int32_t n;
  const uint16_t* in[kNoAllocMaxTensors];
  float* out[kNoAllocMaxTensors];
  int64_t numel[kNoAllocMaxTensors];
  int64_t first_chunk[kNoAllocMaxTensors];
};
static_assert(sizeof(TensorTable) <= 32760, "tensor table must fit in the kernel parameters");

__global__ void noalloc_build_chunks(const __grid_constant__ TensorTable tt, unsigned char* scratch) {
  ListWs* ws = reinterpret_cast<ListWs*>(scratch);
  Chunk* chunks = reinterpret_cast<Chunk*>(scratch + kNoAllocWsBytes);
  if (threadIdx.x == 0) {
    ws->arrived = 0;  // both epilogue words must start at zero
    ws->found = 0;
  }
  for (int t = 0; t < tt.n; ++t) {
    const int64_t n = tt.numel[t], head = chunk_head(tt.in[t], tt.out[t], n);
    const int64_t nc = chunk_count(n, head);
    for (int64_t c = threadIdx.x; c < nc; c += blockDim.x)
      chunks[tt.first_chunk[t] + c] = chunk_at(tt.in[t], tt.out[t], n, head, c);
  }
}

}  // namespace gs

using namespace gs;

extern "C" int gs_noalloc_limits(int32_t* max_tensors, int64_t* max_chunks, int64_t* chunk_elems) {
  if (max_tensors) *max_tensors = kNoAllocMaxTensors;
  if (max_chunks) *max_chunks = kNoAllocMaxChunks;
  if (chunk_elems) *chunk_elems = kChunkElems;
  return GS_OK;
}

extern "C" int gs_unscale_check_update_noalloc(const void* const* grads, void* const* outs,
                                               const int64_t* numels, int32_t n_tensors,
                                               float* scale, int32_t* growth_tracker,
                                               int32_t* found_inf, int64_t* skipped,
                                               float growth_factor, float backoff_factor,
                                               int32_t growth_interval, void* stream) {
  if (!scale || !growth_tracker || !found_inf) return GS_ERR_NULL;
  if (n_tensors < 0 || n_tensors > kNoAllocMaxTensors) return GS_ERR_SHAPE;
  if (n_tensors > 0 && (!grads || !outs || !numels)) return GS_ERR_NULL;
  if (growth_interval < 1) return GS_ERR_ARG;
  if (!std::isfinite(growth_factor) || !(growth_factor > 0.0f) || !std::isfinite(backoff_factor) ||
      !(backoff_factor > 0.0f))
    return GS_ERR_ARG;
  TensorTable tt;
  tt.n = 0;
  int64_t n_chunks = 0;
  for (int32_t i = 0; i < n_tensors; ++i) {
    const int64_t n = numels[i];
    if (n < 0 || n > (INT64_MAX >> 3)) return GS_ERR_SHAPE;
    if (n == 0) continue;
    if (!grads[i] || !outs[i]) return GS_ERR_NULL;
    const int64_t nc = chunk_count(n, chunk_head(static_cast<const uint16_t*>(grads[i]),
                                                 static_cast<const float*>(outs[i]), n));
    if (nc > kNoAllocMaxChunks - n_chunks) return GS_ERR_SHAPE;  // beyond the scratch array
    tt.in[tt.n] = static_cast<const uint16_t*>(grads[i]);
    tt.out[tt.n] = static_cast<float*>(outs[i]);
    tt.numel[tt.n] = n;
    tt.first_chunk[tt.n] = n_chunks;
    ++tt.n;
    n_chunks += nc;
  }
  // The same per-pointer checks as gs_tensor_list_create and
  // gs_unscale_check_update, applied to every pointer; the ranges live on
  // the stack (this entry point allocates nothing).
  Span written[kNoAllocMaxTensors], read[kNoAllocMaxTensors];
  for (int32_t i = 0; i < tt.n; ++i) {
    const int64_t n = tt.numel[i];
    if (((uintptr_t)tt.in[i] & 1u) || ((uintptr_t)tt.out[i] & 3u)) return GS_ERR_ARG;
    const uintptr_t a = (uintptr_t)tt.in[i], b = (uintptr_t)tt.out[i];
    written[i] = Span{b, b + (uintptr_t)n * 4};
    read[i] = Span{a, a + (uintptr_t)n * 2};
    if (!device_reachable(tt.in[i]) || !device_reachable(tt.out[i])) return GS_ERR_ARG;
  }
  // no output may overlap any input or any other output
  if (spans_conflict(written, (size_t)tt.n, read, (size_t)tt.n)) return GS_ERR_ARG;
  if (((uintptr_t)scale & 3u) || ((uintptr_t)growth_tracker & 3u) || ((uintptr_t)found_inf & 3u) ||
      (skipped && ((uintptr_t)skipped & 7u)))
    return GS_ERR_ARG;
  for (const void* p : {(const void*)scale, (const void*)growth_tracker, (const void*)found_inf,
                        (const void*)skipped})
    if (p && !device_reachable(p)) return GS_ERR_ARG;
  // The array's address in the current context: each context that loads
  // the library (each device's primary context, the new primary context
  // after cudaDeviceReset, any context the caller creates) holds its own
  // copy, so the address is looked up per context (symbol_address).
  void* scratch_p = nullptr;
  cudaError_t e = symbol_address((const void*)g_noalloc_scratch, &scratch_p);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return GS_ERR_CUDA;
  }
  unsigned char* scratch = static_cast<unsigned char*>(scratch_p);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  noalloc_build_chunks<<<1, 256, 0, st>>>(tt, scratch);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return GS_ERR_CUDA;
  }
  e = launch_unscale_check_update(reinterpret_cast<const Chunk*>(scratch + kNoAllocWsBytes), n_chunks,
                                  reinterpret_cast<ListWs*>(scratch), scale, growth_tracker,
                                  found_inf, skipped, growth_factor, backoff_factor,
                                  growth_interval, st);
  if (e != cudaSuccess) record_cuda_error(e);
  return e == cudaSuccess ? GS_OK : GS_ERR_CUDA;
}
