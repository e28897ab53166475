// synth.cu — seeded synthetic tensors drawn on the GPU (inputs only).
//
// Holds none of the BitDelta arithmetic: it draws W_base ~ N(0, sigma),
// x ~ N(0, 1) and W_ft = bf16(W_base + Laplace(0, b)) for workloads too large
// to draw on the host.  Random numbers come from a counter-based generator:
// SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014) applied to seed ^ stream-key ^ element index;
// normals by the Box-Muller transform, Laplace deviates by the inverse CDF,
// using the CUDA math library (logf, sincospif, sqrtf).
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace {

__host__ __device__ __forceinline__ uint64_t splitmix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Uniform strictly inside (0, 1): 23 random bits, offset by half a step.  The
// largest value, 1 - 2^-24, is exact in binary32 (with 24 bits the top value
// would round up to 1.0 and the inverse CDFs below would reach log(0)).
__device__ __forceinline__ float u01(uint32_t bits23) {
  return (static_cast<float>(bits23) + 0.5f) * (1.0f / 8388608.0f);
}

__host__ __device__ __forceinline__ uint64_t key(uint64_t seed, uint64_t stream) {
  return splitmix64(seed * 0x632BE59BD9B4E019ull + stream);
}

// Standard normal for element i (one Box-Muller draw per element).
__device__ __forceinline__ float normal_at(uint64_t k, uint64_t i) {
  const uint64_t r = splitmix64(k ^ (i * 0xD1B54A32D192ED03ull));
  const float u1 = u01(static_cast<uint32_t>(r >> 41));
  const float u2 = u01(static_cast<uint32_t>(r >> 8) & 0x7FFFFFu);
  float s, c;
  sincospif(2.0f * u2, &s, &c);
  return sqrtf(-2.0f * logf(u1)) * c;
}

// Laplace(0, b) for element i, inverse CDF.
__device__ __forceinline__ float laplace_at(uint64_t k, uint64_t i, float b) {
  const uint64_t r = splitmix64(k ^ (i * 0xA0761D6478BD642Full));
  const float u = u01(static_cast<uint32_t>(r >> 41)) - 0.5f;
  const float a = fabsf(u);
  const float mag = -b * logf(1.0f - 2.0f * a);
  return u < 0.f ? -mag : mag;
}

__global__ void normal_bf16_kernel(__nv_bfloat16* out, int64_t n, uint64_t k, float sigma) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[i] = __float2bfloat16_rn(sigma * normal_at(k, static_cast<uint64_t>(i)));
}

__global__ void finetuned_bf16_kernel(__nv_bfloat16* out, const __nv_bfloat16* base, int64_t n,
                                      uint64_t k, float b) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[i] = __float2bfloat16_rn(__bfloat162float(base[i]) + laplace_at(k, static_cast<uint64_t>(i), b));
}

int grid_for(int64_t n) {
  const int64_t blocks = (n + 255) / 256;
  return static_cast<int>(blocks < 152 * 16 ? blocks : 152 * 16);
}

}  // namespace

extern "C" {

// out[i] = bf16(sigma * N(0,1)), element i drawn from (seed, stream, i).
int synth_normal_bf16(void* out, int64_t n, uint64_t seed, uint64_t stream, float sigma,
                      void* cuda_stream) {
  if (n <= 0) return 0;
  normal_bf16_kernel<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
      static_cast<__nv_bfloat16*>(out), n, key(seed, stream), sigma);
  return static_cast<int>(cudaGetLastError());
}

// out[i] = bf16(float(base[i]) + Laplace(0, b)).
int synth_finetuned_bf16(void* out, const void* base, int64_t n, uint64_t seed, uint64_t stream,
                         float b, void* cuda_stream) {
  if (n <= 0) return 0;
  finetuned_bf16_kernel<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
      static_cast<__nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(base), n,
      key(seed, stream), b);
  return static_cast<int>(cudaGetLastError());
}

}  // extern "C"
