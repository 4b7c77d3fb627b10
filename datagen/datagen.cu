/*
 * datagen.cu -- host and device fills for the seeded synthetic inputs of
 * dg.h, plus a one-element "plant" used to inject Inf/NaN patterns.
 * Input generation only: none of the cast-and-scale arithmetic lives here.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "dg.h"

extern "C" {

/* out[k] = value of element start + k, for k in [0, n). */
void dg_fill_host(const dg_spec* s, int64_t start, int64_t n, uint16_t* out) {
  for (int64_t k = 0; k < n; ++k) out[k] = dg_value(s, (uint64_t)(start + k));
}

/* out[k] = value of element idx[k]. */
void dg_fill_host_idx(const dg_spec* s, const int64_t* idx, int64_t n, uint16_t* out) {
  for (int64_t k = 0; k < n; ++k) out[k] = dg_value(s, (uint64_t)idx[k]);
}

}  // extern "C"

__global__ void dg_fill_kernel(dg_spec s, int64_t start, int64_t n, uint16_t* out) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += stride)
    out[k] = dg_value(&s, (uint64_t)(start + k));
}

__global__ void dg_plant_kernel(uint16_t* p, uint16_t bits) { *p = bits; }

extern "C" {

/* Device fill of n elements into out (device memory), on `stream`.
 * Returns 0 or the CUDA error code of the launch. */
int dg_fill_device(const dg_spec* s, int64_t start, int64_t n, uint16_t* out, void* stream) {
  if (n <= 0) return 0;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (n + 255) / 256;
  int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 16;
  if (blocks > cap) blocks = cap;
  dg_fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(*s, start, n, out);
  return (int)cudaGetLastError();
}

/* Write one 16-bit pattern into device memory (stream-ordered). */
int dg_plant_device(uint16_t* p, uint16_t bits, void* stream) {
  dg_plant_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(p, bits);
  return (int)cudaGetLastError();
}

int dg_spec_size(void) { return (int)sizeof(dg_spec); }

}  // extern "C"
