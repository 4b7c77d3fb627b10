// gs_layout.h -- the structures and sizes the device kernels are compiled
// against (the chunk tables of gradient and parameter lists, the unscale
// kernel's workspace and scaler policy), kept apart from the host-only
// declarations of gs_internal.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gs {

// One contiguous run of a gradient tensor: at most kChunkElems elements.
// After an optional short head (chunk_head below), chunk starts are
// multiples of kChunkElems from the first element where input and output
// are both 32-byte aligned, so those chunks are aligned too.  A full chunk
// is exactly one pass of a 256-thread CTA moving two 32-byte vectors (16
// FP16 values each) per thread.
struct Chunk {
  const uint16_t* in;  // scaled FP16 gradients
  float* out;          // FP32 unscaled output
  int64_t n;
};
constexpr int64_t kChunkElems = 8192;

// Elements of a tensor before the first element at which both its FP16
// input and its FP32 output are 32-byte aligned, or 0 when there is no such
// element before the end (or the tensor starts aligned).  A list splits
// each tensor as [0, head) -- one short chunk -- and then kChunkElems-element
// chunks from head, so that a tensor placed at any element offset of a flat
// buffer still gets full chunks the kernel's 32-byte path takes.
__host__ __device__ inline int64_t chunk_head(const uint16_t* in, const float* out, int64_t n) {
  const int64_t h = (int64_t)(((32u - ((uint32_t)(uintptr_t)in & 31u)) & 31u) >> 1);
  if (h == 0 || h >= n) return 0;
  return (((uintptr_t)(out + h)) & 31u) == 0 ? h : 0;
}
// Chunks of a tensor of n > 0 elements with that head.
__host__ __device__ inline int64_t chunk_count(int64_t n, int64_t head) {
  return (head > 0 ? 1 : 0) + (n - head + kChunkElems - 1) / kChunkElems;
}
// Chunk c of a tensor of n > 0 elements with that head.
__host__ __device__ inline Chunk chunk_at(const uint16_t* in, float* out, int64_t n, int64_t head,
                                          int64_t c) {
  if (head > 0) {
    if (c == 0) return Chunk{in, out, head};
    --c;
  }
  const int64_t off = head + c * kChunkElems;
  return Chunk{in + off, out + off, (n - off) < kChunkElems ? (n - off) : kChunkElems};
}

// Per-list device workspace of the last-CTA epilogue.  Both words return
// to zero at the end of every call.  A list created by
// gs_tensor_list_create is followed by (SM count) x kUnscaleCtasPerSm double
// slots for the per-CTA sums of squares of the norm-computing form.
struct ListWs {
  unsigned int arrived;
  int32_t found;
  int32_t pad[2];
};
// CTAs per SM of the unscale grid (it walks the chunk table grid-stride):
// several waves, so that CTAs started late even out the SMs' progress;
// measured faster than 32 or 64 and, with the norm's per-CTA slots,
// than 256.
constexpr int kUnscaleCtasPerSm = 128;

// One contiguous run of a parameter tensor for the master-weight update.
struct MChunk {
  float* w;            // fp32 master weights (updated in place)
  uint16_t* w_bf16;    // bf16 copy for the forward pass, or nullptr
  const float* g;      // unscaled fp32 gradients
  int64_t n;
};

// The same split for a parameter tensor: elements before the first element
// at which the fp32 master and gradient are 32-byte aligned and the bf16
// copy (if any) 16-byte aligned -- the master update's vector path -- or 0
// when there is no such element before the end (or the tensor starts
// aligned).
__host__ __device__ inline int64_t mchunk_head(const float* w, const uint16_t* wb,
                                               const float* g, int64_t n) {
  const int64_t h = (int64_t)(((32u - ((uint32_t)(uintptr_t)w & 31u)) & 31u) >> 2);
  if (h == 0 || h >= n) return 0;
  if ((((uintptr_t)(g + h)) & 31u) != 0) return 0;
  if (wb && (((uintptr_t)(wb + h)) & 15u) != 0) return 0;
  return h;
}

// Loss-scale policy applied by the last CTA of the unscale kernel.  With
// hyst == nullptr it is the GradScaler loop; otherwise the hysteresis
// policy: an overflow spends one unit of *hyst (S kept) until one is left,
// then S = max(S * backoff, min_scale); a full clean window grows S and
// restores *hyst (after every clean step when consecutive != 0).
struct ScalerPolicy {
  int32_t* hyst;
  int32_t hysteresis;
  int32_t consecutive;
  float min_scale;
};

}  // namespace gs
