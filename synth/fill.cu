// Device side of the seeded input generator: writes the same bf16 bits as
// synth/gen.py's normal_bits() (splitmix64 output -> top 16 bits -> quantile table).
// Input generation only; nothing here is part of the attention path.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void fill_normal_kernel(uint16_t* __restrict__ out, int64_t count, uint64_t key,
                                   int64_t offset, int log2_scale,
                                   const uint16_t* __restrict__ table) {
  const uint64_t gamma = 0x9E3779B97F4A7C15ull;
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < count; j += stride) {
    uint64_t z = key + (uint64_t)(offset + j + 1) * gamma;
    uint16_t b = __ldg(table + (mix64(z) >> 48));
    out[j] = (uint16_t)(b + (log2_scale << 7));
  }
}

}  // namespace

extern "C" int synth_fill_normal_bf16(void* out, int64_t count, uint64_t key, int64_t offset,
                                      int log2_scale, const void* table, void* stream) {
  if (count <= 0) return 0;
  int blocks = (int)((count + 255) / 256);
  if (blocks > 152 * 32) blocks = 152 * 32;
  fill_normal_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(
      (uint16_t*)out, count, key, offset, log2_scale, (const uint16_t*)table);
  return (int)cudaGetLastError();
}
