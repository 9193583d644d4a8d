/*
 * Device twin of the seeded synthetic input generator (see philox.h).
 * Built as synth/_build/libsynth_dev.so; produces the same bits as
 * synth_fill_host for the same arguments.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include "philox.h"

__global__ void synth_fill_kernel(float* __restrict__ out, int64_t n, uint64_t seed, uint64_t stream,
                                  uint64_t first_index, uint32_t range, int32_t exp2) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    out[i] = synth_sample(seed, stream, first_index + (uint64_t)i, range, exp2);
  }
}

/* Returns a cudaError_t value (0 on success). */
extern "C" int synth_fill_device(float* d_out, int64_t n, uint64_t seed, uint64_t stream,
                                 uint64_t first_index, uint32_t range, int32_t exp2, void* cuda_stream) {
  if (n <= 0) return 0;
  if (d_out == nullptr) return (int)cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return (int)e;
  int64_t blocks = (n + 255) / 256;
  int64_t cap = (int64_t)sms * 16;
  if (blocks > cap) blocks = cap;
  synth_fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)cuda_stream>>>(d_out, n, seed, stream, first_index,
                                                                             range, exp2);
  return (int)cudaGetLastError();
}
