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
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <cmath>
#include <mutex>

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

// The driver's context queries, reached through the runtime (the library
// links no driver library).  Looked up once per process.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
struct CtxQueries {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};
static const CtxQueries& ctx_queries() {
  static CtxQueries q;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &r) ==
            cudaSuccess && r == cudaDriverEntryPointSuccess)
      q.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &r) ==
            cudaSuccess && r == cudaDriverEntryPointSuccess)
      q.get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  return q;
}

// ID of the CUDA context current on this thread, or 0 when there is none.
// The driver never hands out an ID twice in a process, whereas a new
// context may reuse a destroyed one's handle, so the ID is the key.
static bool current_context_id(unsigned long long* id) {
  const CtxQueries& q = ctx_queries();
  CUcontext ctx = nullptr;
  *id = 0;
  if (!q.get_current || !q.get_id || q.get_current(&ctx) != CUDA_SUCCESS) return false;
  return ctx == nullptr || q.get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the CUDA context current on this
// thread.  The array is a module global, so every context that loads the
// library (each device's primary context, the new primary context that
// follows a cudaDeviceReset, any context the caller creates) holds its own
// copy at its own address.  The address is looked up with
// cudaGetSymbolAddress on the first call in a context and cached under the
// context's ID; a call in another context never sees it.
static unsigned char* scratch_address(cudaError_t* err) {
  constexpr int kSlots = 32;
  struct Slot {
    unsigned long long ctx_id;
    unsigned char* ptr;
  };
  static Slot slots[kSlots] = {};
  static int next_slot = 0;
  static std::mutex mu;
  unsigned long long id = 0;
  if (!current_context_id(&id)) {
    *err = cudaErrorDeviceUninitialized;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (id != 0)
    for (const Slot& s : slots)
      if (s.ctx_id == id) {
        *err = cudaSuccess;
        return s.ptr;
      }
  // First call in this context (or no context current yet: the lookup makes
  // the device's primary context current, and its ID is read afterwards).
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) {
    *err = e;
    return nullptr;
  }
  if (id == 0 && (!current_context_id(&id) || id == 0)) {
    *err = cudaErrorDeviceUninitialized;
    return nullptr;
  }
  slots[next_slot] = Slot{id, static_cast<unsigned char*>(p)};
  next_slot = (next_slot + 1) % kSlots;
  *err = cudaSuccess;
  return static_cast<unsigned char*>(p);
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
  cudaError_t e = cudaSuccess;
  unsigned char* scratch = scratch_address(&e);
  if (!scratch) {
    record_cuda_error(e);
    return GS_ERR_CUDA;
  }
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
