/*
 * Device side of the seeded synthetic-input generator (see moegen_core.h).
 * Built with -fmad=false so every float operation rounds exactly as on the host.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include "moegen_core.h"

__global__ void moegen_normal_kernel(uint64_t seed, uint32_t tensor, uint32_t sub, uint64_t start,
                                     uint64_t n, float mean, float stdev, float* __restrict__ out) {
  uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (; t < n; t += stride) out[t] = moegen_normal(seed, tensor, sub, start + t, mean, stdev);
}

/* Asynchronous on `stream`; returns the cudaError_t of the launch. */
extern "C" int moegen_normal_f32_device(uint64_t seed, uint32_t tensor, uint32_t sub, uint64_t start,
                                        uint64_t n, float mean, float stdev, float* out,
                                        cudaStream_t stream) {
  if (n == 0) return 0;
  uint64_t blocks = (n + 255) / 256;
  if (blocks > 152ull * 64ull) blocks = 152ull * 64ull;
  moegen_normal_kernel<<<(unsigned)blocks, 256, 0, stream>>>(seed, tensor, sub, start, n, mean,
                                                              stdev, out);
  return (int)cudaGetLastError();
}
