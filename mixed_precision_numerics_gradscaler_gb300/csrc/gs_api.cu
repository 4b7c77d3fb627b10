// gs_api.cu -- the C ABI declared in include/gsfp8.h: argument validation
// on the host (nothing is launched unless every check passes), the
// gradient-list chunk table, status codes and launch dispatch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <map>
#include <mutex>
#include <new>
#include <tuple>
#include <vector>

#include "gs_internal.h"
#include "gsfp8.h"
#include "gsfp8_test.h"

// The device status word (GS_OK or GS_ERR_TIMEOUT), one per CUDA context.
__device__ int32_t g_gs_device_status = 0;

struct gs_tensor_list {
  int device;
  gs::Chunk* d_chunks;
  int64_t n_chunks;
  int64_t total;
  gs::ListWs* d_ws;       // epilogue words, then the norm slots
  double* d_norm_slots;   // one per CTA of the unscale grid
};

struct gs_param_list {
  int device;
  gs::MChunk* d_chunks;
  int64_t n_chunks;
  int64_t total;
};

namespace gs {

static thread_local int t_last_cuda_error = 0;
constexpr int kMaxDevices = 64;

int current_device() {
  int d = 0;
  cudaGetDevice(&d);
  return d;
}

int sm_count() {
  static std::atomic<int> cache[kMaxDevices] = {};
  const int d = current_device();
  if (d < 0 || d >= kMaxDevices) return 1;
  int n = cache[d].load(std::memory_order_relaxed);
  if (n == 0) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    if (n < 1) n = 1;
    cache[d].store(n, std::memory_order_relaxed);
  }
  return n;
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

bool current_context_id(unsigned long long* id) {
  const CtxQueries& q = ctx_queries();
  CUcontext ctx = nullptr;
  *id = 0;
  if (!q.get_current || !q.get_id || q.get_current(&ctx) != CUDA_SUCCESS) return false;
  return ctx == nullptr || q.get_id(ctx, id) == CUDA_SUCCESS;
}

// ID of the current context, making the device's primary context current
// first when no context is (as the runtime does on its first call).
static cudaError_t context_id(unsigned long long* id) {
  if (!current_context_id(id)) return cudaErrorDeviceUninitialized;
  if (*id != 0) return cudaSuccess;
  const cudaError_t e = cudaFree(nullptr);  // initialises the primary context, frees nothing
  if (e != cudaSuccess) return e;
  return current_context_id(id) && *id != 0 ? cudaSuccess : cudaErrorDeviceUninitialized;
}

cudaError_t symbol_address(const void* symbol, void** out) {
  constexpr int kSlots = 64;
  struct Slot {
    const void* symbol;
    unsigned long long ctx_id;
    void* ptr;
  };
  static Slot slots[kSlots] = {};
  static int next_slot = 0;
  static std::mutex mu;
  *out = nullptr;
  unsigned long long id = 0;
  cudaError_t e = context_id(&id);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (const Slot& sl : slots)
    if (sl.ctx_id == id && sl.symbol == symbol) {
      *out = sl.ptr;
      return cudaSuccess;
    }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, symbol);
  if (e != cudaSuccess) return e;
  slots[next_slot] = Slot{symbol, id, p};
  next_slot = (next_slot + 1) % kSlots;
  *out = p;
  return cudaSuccess;
}

cudaError_t kernel_blocks_per_sm(const void* kernel, int threads, int smem_bytes, int* blocks) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, unsigned long long, int, int>, int> cache;
  unsigned long long ctx = 0;
  const cudaError_t ce = context_id(&ctx);
  if (ce != cudaSuccess) return ce;
  const auto key = std::make_tuple(kernel, ctx, threads, smem_bytes);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it == cache.end()) {
    if (smem_bytes > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           smem_bytes);
      if (e != cudaSuccess) return e;
    }
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, smem_bytes);
    if (e != cudaSuccess) return e;
    it = cache.emplace(key, occ).first;
  }
  *blocks = it->second;
  return cudaSuccess;
}

void record_cuda_error(cudaError_t e) { t_last_cuda_error = (int)e; }

// The status word's address in the current context.
static cudaError_t device_status_ptr(int32_t** out) {
  void* p = nullptr;
  const cudaError_t e = symbol_address((const void*)&g_gs_device_status, &p);
  *out = static_cast<int32_t*>(p);
  return e;
}

static int cuda_fail(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return GS_ERR_CUDA;
}

// A pointer the current device can dereference as it is: device memory of
// this device, managed memory, or mapped (registered) host memory whose
// device address is the host address itself (the kernels are given p, not
// a translated alias).
bool device_reachable(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of the query
    return false;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
      return a.device == current_device();
    case cudaMemoryTypeManaged:
      return true;
    case cudaMemoryTypeHost:
      return a.devicePointer == p;
    default:
      return false;
  }
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return na && nb && x < y + nb && y < x + na;
}

static size_t dtype_size(int dt) { return dt == GS_F32 ? 4 : 2; }
static bool valid_dtype(int dt) { return dt == GS_F16 || dt == GS_BF16 || dt == GS_F32; }
static bool valid_fmt(int f) { return f == GS_E4M3 || f == GS_E5M2; }

static bool mul_ok(int64_t a, int64_t b) { return a >= 0 && b >= 0 && (b == 0 || a <= INT64_MAX / b); }

bool spans_conflict(Span* writes, size_t n_writes, const Span* reads, size_t n_reads) {
  size_t k = 0;  // drop empty ranges
  for (size_t i = 0; i < n_writes; ++i)
    if (writes[i].hi > writes[i].lo) writes[k++] = writes[i];
  std::sort(writes, writes + k, [](const Span& a, const Span& b) { return a.lo < b.lo; });
  for (size_t i = 1; i < k; ++i)
    if (writes[i].lo < writes[i - 1].hi) return true;
  // the written ranges are now disjoint and sorted by both ends: a read range
  // meets one only if it meets the last one starting before its end
  for (size_t i = 0; i < n_reads; ++i) {
    const Span r = reads[i];
    if (r.hi <= r.lo) continue;
    const Span* w = std::lower_bound(writes, writes + k, r.hi,
                                     [](const Span& a, uintptr_t v) { return a.lo < v; });
    if (w != writes && (w - 1)->hi > r.lo) return true;
  }
  return false;
}

static std::atomic<int> g_test_stall{0};
int test_stall() { return g_test_stall.load(std::memory_order_relaxed); }

}  // namespace gs

using namespace gs;

extern "C" {

const char* gs_status_str(int status) {
  switch (status) {
    case GS_OK: return "GS_OK";
    case GS_ERR_NULL: return "GS_ERR_NULL: a required pointer is NULL";
    case GS_ERR_SHAPE: return "GS_ERR_SHAPE: invalid sizes or block shape";
    case GS_ERR_DTYPE: return "GS_ERR_DTYPE: unsupported element type or FP8 format";
    case GS_ERR_ARG: return "GS_ERR_ARG: invalid argument";
    case GS_ERR_CUDA: return "GS_ERR_CUDA: a CUDA call failed";
    case GS_ERR_TIMEOUT: return "GS_ERR_TIMEOUT: a bounded device-side wait expired";
    default: return "unknown gs_status";
  }
}

int gs_last_cuda_error(void) { return t_last_cuda_error; }

const char* gs_version(void) { return "gsfp8 0.1.0 (sm_103a)"; }

int gs_tensor_list_create(const void* const* grads, void* const* outs, const int64_t* numels,
                          int32_t n_tensors, gs_tensor_list** out) {
  if (!out) return GS_ERR_NULL;
  *out = nullptr;
  if (n_tensors < 0) return GS_ERR_SHAPE;
  if (n_tensors > 0 && (!grads || !outs || !numels)) return GS_ERR_NULL;
  std::vector<Chunk> chunks;
  int64_t total = 0;
  try {  // nothing may throw across the C ABI (a vector that cannot grow)
    std::vector<Span> written, read;
    for (int32_t i = 0; i < n_tensors; ++i) {
      const int64_t n = numels[i];
      if (n < 0 || n > (INT64_MAX >> 3) || total > INT64_MAX - n) return GS_ERR_SHAPE;
      if (n == 0) continue;
      if (!grads[i] || !outs[i]) return GS_ERR_NULL;
      if (!aligned(grads[i], 2) || !aligned(outs[i], 4)) return GS_ERR_ARG;
      if (!device_reachable(grads[i]) || !device_reachable(outs[i])) return GS_ERR_ARG;
      written.push_back(Span{(uintptr_t)outs[i], (uintptr_t)outs[i] + (uintptr_t)n * 4});
      read.push_back(Span{(uintptr_t)grads[i], (uintptr_t)grads[i] + (uintptr_t)n * 2});
      const uint16_t* g = static_cast<const uint16_t*>(grads[i]);
      float* o = static_cast<float*>(outs[i]);
      const int64_t head = chunk_head(g, o, n), nc = chunk_count(n, head);
      for (int64_t c = 0; c < nc; ++c) chunks.push_back(chunk_at(g, o, n, head, c));
      total += n;
    }
    // one launch covers every tensor: no output may overlap any input or
    // any other output
    if (spans_conflict(written.data(), written.size(), read.data(), read.size()))
      return GS_ERR_ARG;
  } catch (...) {
    return GS_ERR_ARG;
  }
  gs_tensor_list* l =
      new (std::nothrow) gs_tensor_list{current_device(), nullptr, 0, total, nullptr, nullptr};
  if (!l) return GS_ERR_ARG;
  const size_t ws_bytes = 256 + (size_t)sm_count() * kUnscaleCtasPerSm * sizeof(double);
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&l->d_ws), ws_bytes);
  if (e == cudaSuccess) e = cudaMemsetAsync(l->d_ws, 0, ws_bytes, cudaStreamLegacy);
  l->d_norm_slots = reinterpret_cast<double*>(reinterpret_cast<char*>(l->d_ws) + 256);
  if (e == cudaSuccess && !chunks.empty()) {
    e = cudaMalloc(reinterpret_cast<void**>(&l->d_chunks), chunks.size() * sizeof(Chunk));
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(l->d_chunks, chunks.data(), chunks.size() * sizeof(Chunk),
                          cudaMemcpyHostToDevice, cudaStreamLegacy);
  }
  // Both must have landed before the call returns: a step launched next on a
  // non-blocking stream is not ordered behind the legacy stream, and a copy
  // from pageable memory may return before its data reaches the device.
  if (e == cudaSuccess) e = cudaStreamSynchronize(cudaStreamLegacy);
  if (e != cudaSuccess) {
    if (l->d_chunks) cudaFree(l->d_chunks);
    if (l->d_ws) cudaFree(l->d_ws);
    delete l;
    return cuda_fail(e);
  }
  l->n_chunks = (int64_t)chunks.size();
  *out = l;
  return GS_OK;
}

int gs_tensor_list_destroy(gs_tensor_list* list) {
  if (!list) return GS_OK;
  int prev = current_device();
  cudaSetDevice(list->device);
  cudaError_t e = cudaDeviceSynchronize();
  if (list->d_chunks) cudaFree(list->d_chunks);
  if (list->d_ws) cudaFree(list->d_ws);
  cudaSetDevice(prev);
  delete list;
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

int gs_tensor_list_info(const gs_tensor_list* list, int64_t* total_elems, int64_t* n_chunks) {
  if (!list) return GS_ERR_NULL;
  if (total_elems) *total_elems = list->total;
  if (n_chunks) *n_chunks = list->n_chunks;
  return GS_OK;
}

int gs_unscale_check_update(const gs_tensor_list* list, float* scale, int32_t* growth_tracker,
                            int32_t* found_inf, int64_t* skipped, float growth_factor,
                            float backoff_factor, int32_t growth_interval, void* stream) {
  if (!list || !scale || !growth_tracker || !found_inf) return GS_ERR_NULL;
  if (growth_interval < 1) return GS_ERR_ARG;
  if (!std::isfinite(growth_factor) || !(growth_factor > 0.0f) || !std::isfinite(backoff_factor) ||
      !(backoff_factor > 0.0f))
    return GS_ERR_ARG;
  if (list->device != current_device()) return GS_ERR_ARG;
  if (!aligned(scale, 4) || !aligned(growth_tracker, 4) || !aligned(found_inf, 4) ||
      (skipped && !aligned(skipped, 8)))
    return GS_ERR_ARG;
  if (!device_reachable(scale) || !device_reachable(growth_tracker) || !device_reachable(found_inf) ||
      (skipped && !device_reachable(skipped)))
    return GS_ERR_ARG;
  cudaError_t e = launch_unscale_check_update(list->d_chunks, list->n_chunks, list->d_ws, scale,
                                              growth_tracker, found_inf, skipped, growth_factor,
                                              backoff_factor, growth_interval,
                                              static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

int gs_unscale_check_update_norm(const gs_tensor_list* list, float* scale, int32_t* growth_tracker,
                                 int32_t* found_inf, int64_t* skipped, float growth_factor,
                                 float backoff_factor, int32_t growth_interval, float* grad_norm,
                                 void* stream) {
  if (!list || !scale || !growth_tracker || !found_inf || !grad_norm) return GS_ERR_NULL;
  if (growth_interval < 1) return GS_ERR_ARG;
  if (!std::isfinite(growth_factor) || !(growth_factor > 0.0f) || !std::isfinite(backoff_factor) ||
      !(backoff_factor > 0.0f))
    return GS_ERR_ARG;
  if (list->device != current_device()) return GS_ERR_ARG;
  if (!aligned(scale, 4) || !aligned(growth_tracker, 4) || !aligned(found_inf, 4) ||
      !aligned(grad_norm, 4) || (skipped && !aligned(skipped, 8)))
    return GS_ERR_ARG;
  if (!device_reachable(scale) || !device_reachable(growth_tracker) || !device_reachable(found_inf) ||
      !device_reachable(grad_norm) || (skipped && !device_reachable(skipped)))
    return GS_ERR_ARG;
  cudaError_t e = launch_unscale_check_update(
      list->d_chunks, list->n_chunks, list->d_ws, scale, growth_tracker, found_inf, skipped,
      growth_factor, backoff_factor, growth_interval, static_cast<cudaStream_t>(stream),
      ScalerPolicy{nullptr, 1, 0, 0.0f}, grad_norm, list->d_norm_slots);
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

int gs_param_list_create(float* const* master, uint16_t* const* master_bf16,
                         const float* const* grads, const int64_t* numels, int32_t n_tensors,
                         gs_param_list** out) {
  if (!out) return GS_ERR_NULL;
  *out = nullptr;
  if (n_tensors < 0) return GS_ERR_SHAPE;
  if (n_tensors > 0 && (!master || !grads || !numels)) return GS_ERR_NULL;
  std::vector<MChunk> chunks;
  int64_t total = 0;
  try {  // nothing may throw across the C ABI (a vector that cannot grow)
    std::vector<Span> written, read;
    for (int32_t i = 0; i < n_tensors; ++i) {
      const int64_t n = numels[i];
      if (n < 0 || n > (INT64_MAX >> 3) || total > INT64_MAX - n) return GS_ERR_SHAPE;
      if (n == 0) continue;
      uint16_t* wb = master_bf16 ? master_bf16[i] : nullptr;
      if (!master[i] || !grads[i]) return GS_ERR_NULL;
      if (!aligned(master[i], 4) || !aligned(grads[i], 4) || (wb && !aligned(wb, 2)))
        return GS_ERR_ARG;
      if (!device_reachable(master[i]) || !device_reachable(grads[i]) ||
          (wb && !device_reachable(wb)))
        return GS_ERR_ARG;
      written.push_back(Span{(uintptr_t)master[i], (uintptr_t)master[i] + (uintptr_t)n * 4});
      if (wb) written.push_back(Span{(uintptr_t)wb, (uintptr_t)wb + (uintptr_t)n * 2});
      read.push_back(Span{(uintptr_t)grads[i], (uintptr_t)grads[i] + (uintptr_t)n * 4});
      // a short head chunk up to the first element where the vector path's
      // alignments hold, then full chunks from there
      const int64_t head = mchunk_head(master[i], wb, grads[i], n);
      if (head > 0) chunks.push_back(MChunk{master[i], wb, grads[i], head});
      for (int64_t off = head; off < n; off += kChunkElems)
        chunks.push_back(MChunk{master[i] + off, wb ? wb + off : nullptr, grads[i] + off,
                                (n - off) < kChunkElems ? (n - off) : kChunkElems});
      total += n;
    }
    // masters and bf16 copies are written: none may overlap another one or a
    // gradient
    if (spans_conflict(written.data(), written.size(), read.data(), read.size()))
      return GS_ERR_ARG;
  } catch (...) {
    return GS_ERR_ARG;
  }
  gs_param_list* l = new (std::nothrow) gs_param_list{current_device(), nullptr, 0, total};
  if (!l) return GS_ERR_ARG;
  cudaError_t e = cudaSuccess;
  if (!chunks.empty()) {
    e = cudaMalloc(reinterpret_cast<void**>(&l->d_chunks), chunks.size() * sizeof(MChunk));
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(l->d_chunks, chunks.data(), chunks.size() * sizeof(MChunk),
                          cudaMemcpyHostToDevice, cudaStreamLegacy);
    // landed before the call returns (as for gradient lists)
    if (e == cudaSuccess) e = cudaStreamSynchronize(cudaStreamLegacy);
  }
  if (e != cudaSuccess) {
    if (l->d_chunks) cudaFree(l->d_chunks);
    delete l;
    return cuda_fail(e);
  }
  l->n_chunks = (int64_t)chunks.size();
  *out = l;
  return GS_OK;
}

int gs_param_list_destroy(gs_param_list* list) {
  if (!list) return GS_OK;
  int prev = current_device();
  cudaSetDevice(list->device);
  cudaError_t e = cudaDeviceSynchronize();
  if (list->d_chunks) cudaFree(list->d_chunks);
  cudaSetDevice(prev);
  delete list;
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

int gs_master_update_sgd(const gs_param_list* list, float lr, float max_norm,
                         const float* grad_norm, const int32_t* found_inf, void* stream) {
  if (!list || !found_inf || (max_norm > 0.0f && !grad_norm)) return GS_ERR_NULL;
  if (!std::isfinite(lr) || !std::isfinite(max_norm)) return GS_ERR_ARG;
  if (list->device != current_device()) return GS_ERR_ARG;
  if (!aligned(found_inf, 4) || (grad_norm && !aligned(grad_norm, 4))) return GS_ERR_ARG;
  if (!device_reachable(found_inf) || (grad_norm && !device_reachable(grad_norm))) return GS_ERR_ARG;
  cudaError_t e = launch_master_update_sgd(list->d_chunks, list->n_chunks, lr, max_norm,
                                           grad_norm, found_inf, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

int gs_unscale_check_update_hysteresis(const gs_tensor_list* list, float* scale,
                                       int32_t* growth_tracker, int32_t* hysteresis_state,
                                       int32_t* found_inf, int64_t* skipped, float growth_factor,
                                       float backoff_factor, int32_t window, int32_t hysteresis,
                                       int32_t consecutive_hysteresis, float min_scale,
                                       void* stream) {
  if (!list || !scale || !growth_tracker || !hysteresis_state || !found_inf) return GS_ERR_NULL;
  if (window < 1 || hysteresis < 1) return GS_ERR_ARG;
  if (!std::isfinite(growth_factor) || !(growth_factor > 0.0f) || !std::isfinite(backoff_factor) ||
      !(backoff_factor > 0.0f) || !std::isfinite(min_scale) || min_scale < 0.0f)
    return GS_ERR_ARG;
  if (list->device != current_device()) return GS_ERR_ARG;
  if (!aligned(scale, 4) || !aligned(growth_tracker, 4) || !aligned(hysteresis_state, 4) ||
      !aligned(found_inf, 4) || (skipped && !aligned(skipped, 8)))
    return GS_ERR_ARG;
  if (!device_reachable(scale) || !device_reachable(growth_tracker) ||
      !device_reachable(hysteresis_state) || !device_reachable(found_inf) ||
      (skipped && !device_reachable(skipped)))
    return GS_ERR_ARG;
  cudaError_t e = launch_unscale_check_update(
      list->d_chunks, list->n_chunks, list->d_ws, scale, growth_tracker, found_inf, skipped,
      growth_factor, backoff_factor, window, static_cast<cudaStream_t>(stream),
      ScalerPolicy{hysteresis_state, hysteresis, consecutive_hysteresis ? 1 : 0, min_scale});
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

int gs_scaler_state_get(const float* scale, const int32_t* growth_tracker, float* h_scale,
                        int32_t* h_growth_tracker, void* stream) {
  if (!scale || !growth_tracker || !h_scale || !h_growth_tracker) return GS_ERR_NULL;
  if (!device_reachable(scale) || !device_reachable(growth_tracker)) return GS_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(h_scale, scale, sizeof(float), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(h_growth_tracker, growth_tracker, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

int gs_scaler_state_set(float* scale, int32_t* growth_tracker, float h_scale,
                        int32_t h_growth_tracker, void* stream) {
  if (!scale || !growth_tracker) return GS_ERR_NULL;
  if (h_growth_tracker < 0) return GS_ERR_ARG;
  if (!device_reachable(scale) || !device_reachable(growth_tracker)) return GS_ERR_ARG;
  cudaError_t e = launch_set_state(scale, growth_tracker, h_scale, h_growth_tracker,
                                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

int fp8_quant_block(const void* x, int in_dtype, int64_t R, int64_t C, int32_t block_r,
                    int32_t block_c, int fmt, uint8_t* q, float* scales, void* stream) {
  if (!valid_dtype(in_dtype) || !valid_fmt(fmt)) return GS_ERR_DTYPE;
  if (R < 0 || C < 0 || !mul_ok(R, C) || !mul_ok(R * C, 4)) return GS_ERR_SHAPE;
  if (!((block_r == 1 || block_r == 128) && block_c == 128)) return GS_ERR_SHAPE;
  if (R % block_r != 0 || C % block_c != 0) return GS_ERR_SHAPE;
  if (R == 0 || C == 0) return GS_OK;
  if (!x || !q || !scales) return GS_ERR_NULL;
  const size_t n = (size_t)(R * C), esz = dtype_size(in_dtype);
  const size_t nscales = (size_t)((R / block_r) * (C / block_c));
  if (!aligned(x, esz) || !aligned(scales, 4)) return GS_ERR_ARG;
  if (!device_reachable(x) || !device_reachable(q) || !device_reachable(scales)) return GS_ERR_ARG;
  if (overlaps(x, n * esz, q, n) || overlaps(x, n * esz, scales, nscales * 4) ||
      overlaps(q, n, scales, nscales * 4))
    return GS_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = block_r == 1
                      ? launch_quant_1x128(x, in_dtype, R, C, fmt, q, scales, st)
                      : launch_quant_128x128(x, in_dtype, R, C, fmt, q, scales, st);
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

size_t gs_ws_bytes(void) { return (size_t)kMaxAmaxBlocks * sizeof(uint32_t); }

int fp8_quant_tensor(const void* x, int in_dtype, int64_t n, int fmt, uint8_t* q, float* scale,
                     void* ws, void* stream) {
  if (!valid_dtype(in_dtype) || !valid_fmt(fmt)) return GS_ERR_DTYPE;
  if (n < 0 || !mul_ok(n, 4)) return GS_ERR_SHAPE;
  if (!scale || !ws || (n > 0 && (!x || !q))) return GS_ERR_NULL;
  const size_t esz = dtype_size(in_dtype);
  if (!aligned(scale, 4) || !aligned(ws, 4) || (n > 0 && !aligned(x, esz))) return GS_ERR_ARG;
  if (!device_reachable(scale) || !device_reachable(ws) ||
      (n > 0 && (!device_reachable(x) || !device_reachable(q))))
    return GS_ERR_ARG;
  if (overlaps(x, (size_t)n * esz, q, (size_t)n) || overlaps(ws, gs_ws_bytes(), x, (size_t)n * esz) ||
      overlaps(ws, gs_ws_bytes(), q, (size_t)n) || overlaps(scale, 4, q, (size_t)n) ||
      overlaps(scale, 4, x, (size_t)n * esz) || overlaps(scale, 4, ws, gs_ws_bytes()))
    return GS_ERR_ARG;
  cudaError_t e = launch_quant_tensor(x, in_dtype, n, fmt, q, scale, static_cast<uint32_t*>(ws),
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

int fp8_dequant(const uint8_t* q, const float* scales, int64_t R, int64_t C, int32_t block_r,
                int32_t block_c, int fmt, int out_dtype, void* y, void* stream) {
  if (!valid_fmt(fmt) || !(out_dtype == GS_F32 || out_dtype == GS_BF16)) return GS_ERR_DTYPE;
  if (R < 0 || C < 0 || !mul_ok(R, C) || !mul_ok(R * C, 4)) return GS_ERR_SHAPE;
  const bool per_tensor = (int64_t)block_r == R && (int64_t)block_c == C;
  const bool blocked = (block_r == 1 || block_r == 128) && block_c == 128;
  if (!per_tensor && !blocked) return GS_ERR_SHAPE;
  if (!per_tensor && (R % block_r != 0 || C % block_c != 0)) return GS_ERR_SHAPE;
  if (R == 0 || C == 0) return GS_OK;
  if (!q || !scales || !y) return GS_ERR_NULL;
  const size_t n = (size_t)(R * C), ysz = out_dtype == GS_F32 ? 4 : 2;
  const size_t nscales = per_tensor ? 1 : (size_t)((R / block_r) * (C / block_c));
  if (!aligned(scales, 4) || !aligned(y, ysz)) return GS_ERR_ARG;
  if (!device_reachable(q) || !device_reachable(scales) || !device_reachable(y)) return GS_ERR_ARG;
  if (overlaps(y, n * ysz, q, n) || overlaps(y, n * ysz, scales, nscales * 4)) return GS_ERR_ARG;
  cudaError_t e = launch_dequant(q, scales, R, C, block_r, block_c, fmt, out_dtype, y,
                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

int fp8_quant_tensor_delayed(const void* x, int in_dtype, int64_t n, int fmt, uint8_t* q,
                             float* amax_history, int32_t history_len, int32_t* history_pos,
                             float* scale_used, void* ws, void* stream) {
  if (!valid_dtype(in_dtype) || !valid_fmt(fmt)) return GS_ERR_DTYPE;
  if (n < 0 || !mul_ok(n, 4)) return GS_ERR_SHAPE;
  if (history_len < 1 || history_len > 65536) return GS_ERR_ARG;
  if (!amax_history || !history_pos || !scale_used || !ws || (n > 0 && (!x || !q)))
    return GS_ERR_NULL;
  const size_t esz = dtype_size(in_dtype), hb = (size_t)history_len * 4;
  if (!aligned(amax_history, 4) || !aligned(history_pos, 4) || !aligned(scale_used, 4) ||
      !aligned(ws, 4) || (n > 0 && !aligned(x, esz)))
    return GS_ERR_ARG;
  if (!device_reachable(amax_history) || !device_reachable(history_pos) ||
      !device_reachable(scale_used) || !device_reachable(ws) ||
      (n > 0 && (!device_reachable(x) || !device_reachable(q))))
    return GS_ERR_ARG;
  const size_t xb = (size_t)n * esz, wb = gs_ws_bytes();
  if (overlaps(x, xb, q, (size_t)n) || overlaps(amax_history, hb, q, (size_t)n) ||
      overlaps(amax_history, hb, x, xb) || overlaps(ws, wb, x, xb) || overlaps(ws, wb, q, (size_t)n) ||
      overlaps(ws, wb, amax_history, hb) || overlaps(scale_used, 4, q, (size_t)n) ||
      overlaps(scale_used, 4, amax_history, hb) || overlaps(history_pos, 4, amax_history, hb))
    return GS_ERR_ARG;
  cudaError_t e = launch_quant_tensor_delayed(x, in_dtype, n, fmt, q, amax_history, history_len,
                                              history_pos, scale_used, static_cast<uint32_t*>(ws),
                                              static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

int fp8_quant_mx(const void* x, int in_dtype, int64_t R, int64_t C, int fmt, uint8_t* q,
                 uint8_t* scales, void* stream) {
  if (!valid_dtype(in_dtype) || !valid_fmt(fmt)) return GS_ERR_DTYPE;
  if (R < 0 || C < 0 || !mul_ok(R, C) || !mul_ok(R * C, 4)) return GS_ERR_SHAPE;
  if (C % 32 != 0) return GS_ERR_SHAPE;
  if (R == 0 || C == 0) return GS_OK;
  if (!x || !q || !scales) return GS_ERR_NULL;
  const size_t n = (size_t)(R * C), esz = dtype_size(in_dtype), ns = n / 32;
  if (!aligned(x, esz)) return GS_ERR_ARG;
  if (!device_reachable(x) || !device_reachable(q) || !device_reachable(scales)) return GS_ERR_ARG;
  if (overlaps(x, n * esz, q, n) || overlaps(x, n * esz, scales, ns) || overlaps(q, n, scales, ns))
    return GS_ERR_ARG;
  cudaError_t e = launch_quant_mx(x, in_dtype, R, C, fmt, q, scales, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

int fp8_dequant_mx(const uint8_t* q, const uint8_t* scales, int64_t R, int64_t C, int fmt,
                   int out_dtype, void* y, void* stream) {
  if (!valid_fmt(fmt) || !(out_dtype == GS_F32 || out_dtype == GS_BF16)) return GS_ERR_DTYPE;
  if (R < 0 || C < 0 || !mul_ok(R, C) || !mul_ok(R * C, 4)) return GS_ERR_SHAPE;
  if (C % 32 != 0) return GS_ERR_SHAPE;
  if (R == 0 || C == 0) return GS_OK;
  if (!q || !scales || !y) return GS_ERR_NULL;
  const size_t n = (size_t)(R * C), ysz = out_dtype == GS_F32 ? 4 : 2;
  if (!aligned(y, ysz)) return GS_ERR_ARG;
  if (!device_reachable(q) || !device_reachable(scales) || !device_reachable(y)) return GS_ERR_ARG;
  if (overlaps(y, n * ysz, q, n) || overlaps(y, n * ysz, scales, n / 32)) return GS_ERR_ARG;
  cudaError_t e = launch_dequant_mx(q, scales, R, C, fmt, out_dtype, y,
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

int fp8_gemm_block_scaled(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                          int64_t M, int64_t N, int64_t K, int fmt_a, int fmt_b, int out_dtype,
                          void* d, void* stream) {
  if (!valid_fmt(fmt_a) || !valid_fmt(fmt_b) || !(out_dtype == GS_F32 || out_dtype == GS_BF16))
    return GS_ERR_DTYPE;
  if (M < 0 || N < 0 || K < 0 || K % 128 != 0 || M >= (1LL << 31) || K >= (1LL << 31) ||
      N >= (1LL << 31) || !mul_ok(M, N) || !mul_ok(M * N, 4) || !mul_ok(M, K) || !mul_ok(N, K))
    return GS_ERR_SHAPE;
  if (((M + 127) / 128) * ((N + 255) / 256) >= (1LL << 30)) return GS_ERR_SHAPE;  // tile count
  if (M == 0 || N == 0) return GS_OK;
  if (!d || (K > 0 && (!qa || !sa || !qb || !sb))) return GS_ERR_NULL;
  const size_t dsz = out_dtype == GS_F32 ? 4 : 2, nd = (size_t)(M * N) * dsz;
  if (!aligned(d, dsz)) return GS_ERR_ARG;
  if (!device_reachable(d)) return GS_ERR_ARG;
  if (K > 0) {
    const int64_t nkb = K / 128;
    const size_t na = (size_t)(M * K), nb = (size_t)(N * K);
    const size_t nsa = (size_t)(M * nkb) * 4, nsb = (size_t)(((N + 127) / 128) * nkb) * 4;
    if (!aligned(qa, 16) || !aligned(qb, 16) || !aligned(sa, 4) || !aligned(sb, 4))
      return GS_ERR_ARG;
    if (!device_reachable(qa) || !device_reachable(sa) || !device_reachable(qb) ||
        !device_reachable(sb))
      return GS_ERR_ARG;
    if (overlaps(d, nd, qa, na) || overlaps(d, nd, qb, nb) || overlaps(d, nd, sa, nsa) ||
        overlaps(d, nd, sb, nsb))
      return GS_ERR_ARG;
  }
  int32_t* status = nullptr;
  cudaError_t e = device_status_ptr(&status);
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch_gemm_fp8_block_scaled(qa, sa, qb, sb, M, N, K, fmt_a, fmt_b, out_dtype, d,
                                               status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

int gs_test_set_stall(int on) {
  g_test_stall.store(on ? 1 : 0, std::memory_order_relaxed);
  return GS_OK;
}

int gs_device_status(int32_t* h_status, void* stream) {
  if (!h_status) return GS_ERR_NULL;
  int32_t* p = nullptr;
  cudaError_t e = device_status_ptr(&p);
  if (e != cudaSuccess) return cuda_fail(e);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  e = cudaMemcpyAsync(h_status, p, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, sizeof(int32_t), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e == cudaSuccess ? GS_OK : cuda_fail(e);
}

}  // extern "C"
