// Device generator of synthetic weight planes (see include/moe_gen.h for the definition).
// It holds none of the MoE computation; it reproduces the host generator bit for bit.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe_gen.h"

namespace {

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

__device__ __forceinline__ uint64_t stream_key(uint64_t seed, int layer, int tensor, int expert) {
  uint64_t k = mix64(seed);
  k = mix64(k ^ ((uint64_t)(layer + 1) * 0x9E3779B97F4A7C15ull));
  k = mix64(k ^ ((uint64_t)(tensor + 1) * 0xD1B54A32D192ED03ull));
  k = mix64(k ^ ((uint64_t)(expert + 1) * 0x8CB92BA72F3D8DD7ull));
  return k;
}

// grid: (blocks per expert, n_experts)
__global__ void gen_int4_kernel(uint64_t* dst, uint64_t seed, int layer, int tensor, int expert0, size_t words) {
  const int e = expert0 + blockIdx.y;
  const uint64_t key = stream_key(seed, layer, tensor, e);
  uint64_t* out = dst + (size_t)blockIdx.y * words;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < words; i += (size_t)gridDim.x * blockDim.x)
    out[i] = mix64(key + (uint64_t)(i + 1) * 0x9E3779B97F4A7C15ull);
}

__global__ void gen_scale_kernel(__half* dst, uint64_t seed, int layer, int tensor, int expert0, size_t n) {
  const int e = expert0 + blockIdx.y;
  const uint64_t key = stream_key(seed, layer, tensor, e);
  __half* out = dst + (size_t)blockIdx.y * n;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const uint64_t z = mix64(key + (uint64_t)(i + 1) * 0x9E3779B97F4A7C15ull);
    const double u = (double)(z >> 11) * 0x1.0p-53;
    const double s = __dadd_rn(0.005, __dmul_rn(0.015, u));
    out[i] = __double2half(s);
  }
}

}  // namespace

extern "C" int moe_gen_int4_planes(void* dst, uint64_t seed, int layer, int tensor, int expert0, int n_experts,
                                   size_t bytes_per_expert, void* stream) {
  if (!dst || n_experts <= 0 || n_experts > 65535 || bytes_per_expert % 8 || (reinterpret_cast<uintptr_t>(dst) & 7))
    return 1;
  const size_t words = bytes_per_expert / 8;
  int bx = (int)((words + 255) / 256);
  if (bx > 64) bx = 64;
  gen_int4_kernel<<<dim3(bx, n_experts), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint64_t*>(dst), seed, layer, tensor, expert0, words);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

extern "C" int moe_gen_scale_planes(void* dst, uint64_t seed, int layer, int tensor, int expert0, int n_experts,
                                    size_t scales_per_expert, void* stream) {
  if (!dst || n_experts <= 0 || n_experts > 65535 || (reinterpret_cast<uintptr_t>(dst) & 1)) return 1;
  int bx = (int)((scales_per_expert + 255) / 256);
  if (bx > 64) bx = 64;
  gen_scale_kernel<<<dim3(bx, n_experts), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<__half*>(dst), seed, layer, tensor, expert0, scales_per_expert);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
