// Seeded synthetic inputs on the device: the counter-based SplitMix64 stream
// and the Irwin-Hall bf16 normal draw declared in include/dllm_synth.h.
// Every step is an integer operation or one correctly rounded float32
// operation (__fmul_rn / __fadd_rn, no contraction), so the output bits equal
// the numpy generator's.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/dllm_synth.h"

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t word(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1ull) * 0x9E3779B97F4A7C15ull);
}

__global__ void fill_normal_kernel(uint16_t* dst, int64_t count, uint64_t key, float c, float offset,
                                   int64_t first) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x) {
    uint64_t u = word(key, (uint64_t)(first + i));
    int64_t s = (int64_t)(u & 0xFFFF) + (int64_t)((u >> 16) & 0xFFFF) + (int64_t)((u >> 32) & 0xFFFF) +
                (int64_t)(u >> 48);
    float z = (float)(s - 131070);            // exact: |z| < 2^24
    float w = __fmul_rn(z, c);
    if (offset != 0.0f) w = __fadd_rn(w, offset);
    __nv_bfloat16 b = __float2bfloat16_rn(w);
    dst[i] = *reinterpret_cast<uint16_t*>(&b);
  }
}

__global__ void fill_const_kernel(uint16_t* dst, int64_t count, uint16_t value) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = value;
}

__global__ void fill_ids_kernel(int32_t* dst, int64_t count, uint64_t key, int32_t vocab, int64_t first) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count;
       i += (int64_t)gridDim.x * blockDim.x) {
    uint64_t u = word(key, (uint64_t)(first + i));
    dst[i] = (int32_t)(((u >> 32) * (uint64_t)vocab) >> 32);
  }
}

int grid_for(int64_t count) {
  int64_t g = (count + 255) / 256;
  if (g > 8192) g = 8192;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

extern "C" int dllm_synth_fill_normal_bf16(uint16_t* dst, int64_t count, uint64_t key, float c, float offset,
                                           int64_t first, void* stream) {
  if (count <= 0) return 0;
  fill_normal_kernel<<<grid_for(count), 256, 0, (cudaStream_t)stream>>>(dst, count, key, c, offset, first);
  return (int)cudaGetLastError();
}

extern "C" int dllm_synth_fill_const_bf16(uint16_t* dst, int64_t count, uint16_t value, void* stream) {
  if (count <= 0) return 0;
  fill_const_kernel<<<grid_for(count), 256, 0, (cudaStream_t)stream>>>(dst, count, value);
  return (int)cudaGetLastError();
}

extern "C" int dllm_synth_fill_ids(int32_t* dst, int64_t count, uint64_t key, int32_t vocab, int64_t first,
                                   void* stream) {
  if (count <= 0) return 0;
  fill_ids_kernel<<<grid_for(count), 256, 0, (cudaStream_t)stream>>>(dst, count, key, vocab, first);
  return (int)cudaGetLastError();
}
