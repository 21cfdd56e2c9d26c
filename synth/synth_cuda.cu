// Device fill for the synthetic input generator defined in synth_def.h: the
// same per-element function as the host fill, so host and device produce the
// same bits for the same (seed, tensor id, flat index).
#include <cuda_runtime.h>
#include <stdint.h>
#include "synth_def.h"

__global__ void synth_normal_kernel(uint16_t* __restrict__ out, uint64_t key,
                                    uint64_t start, uint64_t count, double scale_sqrt3) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < count; j += stride)
    out[j] = synth_normal_bf16(key, start + j, scale_sqrt3);
}

__global__ void synth_uniform_kernel(int32_t* __restrict__ out, uint64_t key,
                                     uint64_t start, uint64_t count, uint32_t n) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < count; j += stride)
    out[j] = synth_uniform_int(key, start + j, n);
}

static unsigned grid_for(uint64_t count) {
  uint64_t blocks = (count + 255) / 256;
  if (blocks > 152ull * 16) blocks = 152ull * 16;
  if (blocks == 0) blocks = 1;
  return (unsigned)blocks;
}

extern "C" int synth_fill_normal_bf16_dev(void* out, uint64_t seed, uint64_t tensor_id,
                                          uint64_t start, uint64_t count, double scale_sqrt3,
                                          void* stream) {
  if (count == 0) return 0;
  synth_normal_kernel<<<grid_for(count), 256, 0, (cudaStream_t)stream>>>(
      (uint16_t*)out, synth_key(seed, tensor_id), start, count, scale_sqrt3);
  return (int)cudaGetLastError();
}

extern "C" int synth_fill_uniform_i32_dev(void* out, uint64_t seed, uint64_t tensor_id,
                                          uint64_t start, uint64_t count, uint32_t n,
                                          void* stream) {
  if (count == 0) return 0;
  synth_uniform_kernel<<<grid_for(count), 256, 0, (cudaStream_t)stream>>>(
      (int32_t*)out, synth_key(seed, tensor_id), start, count, n);
  return (int)cudaGetLastError();
}
