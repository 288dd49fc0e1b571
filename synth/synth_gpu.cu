// Seeded synthetic input generator (device side).
//
// Same definition as synth.c (SplitMix64 output function as the counter
// hash, Irwin-Hall(12) in int32, one fp32 multiply, bf16 round-to-nearest-even
// by integer arithmetic), so device-generated tensors equal the host ones bit
// for bit.  It generates inputs only and holds none of the MoE layer's
// arithmetic.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

__device__ __forceinline__ int32_t lanes_sum(uint64_t w) {
  return (int32_t)(w & 0xFFFF) + (int32_t)((w >> 16) & 0xFFFF) +
         (int32_t)((w >> 32) & 0xFFFF) + (int32_t)(w >> 48);
}

__global__ void normal_bf16_kernel(uint16_t* __restrict__ out, uint64_t n, uint64_t offset,
                                   uint64_t stream, float scale) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    uint64_t base = stream + 3 * (offset + i);
    int32_t s = lanes_sum(mix64(base)) + lanes_sum(mix64(base + 1)) + lanes_sum(mix64(base + 2)) - 393210;
    float v = __fmul_rn((float)s, scale);
    uint32_t u = __float_as_uint(v);
    u += 0x7FFFu + ((u >> 16) & 1u);
    out[i] = (uint16_t)(u >> 16);
  }
}

uint64_t host_mix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

}  // namespace

extern "C" int synth_normal_bf16_gpu(void* out, uint64_t n, uint64_t offset, uint64_t seed,
                                     uint64_t tensor_id, float scale, void* stream) {
  if (n == 0) return 0;
  if (out == nullptr) return 1;
  uint64_t s = host_mix64(host_mix64(seed) ^ tensor_id);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  uint64_t want = (n + 255) / 256;
  uint64_t cap = (uint64_t)(sms > 0 ? sms : 1) * 16;
  unsigned grid = (unsigned)(want < cap ? want : cap);
  normal_bf16_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>((uint16_t*)out, n, offset, s, scale);
  return (int)cudaGetLastError();
}
