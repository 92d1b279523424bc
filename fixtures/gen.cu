// Device-side implementation of the fixture generator defined in
// fixtures/__init__.py (SplitMix64 words, Box-Muller normals in float64,
// rounded to float32 and then to bfloat16). Fills the 8B / 70B-shaped weights
// in place on the GPU; the oracle draws the same numbers with numpy.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ double std_normal(uint64_t key, uint64_t i) {
  const uint64_t a = mix64(key + (2 * i + 1) * kGamma);
  const uint64_t b = mix64(key + (2 * i + 2) * kGamma);
  const double u1 = (double)((a >> 11) + 1) * (1.0 / 9007199254740992.0);
  const double u2 = (double)(b >> 11) * (1.0 / 9007199254740992.0);
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

__global__ void fill_normal_kernel(void* dst, int bf16, int64_t count, int64_t start, uint64_t key, double sd,
                                   uint64_t nkey, double nsd, int noise) {
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < count;
       e += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t i = (uint64_t)(start + e);
    double v = sd * std_normal(key, i);
    if (noise) v = v + nsd * std_normal(nkey, i);
    const float f = (float)v;
    if (bf16)
      reinterpret_cast<__nv_bfloat16*>(dst)[e] = __float2bfloat16_rn(f);
    else
      reinterpret_cast<float*>(dst)[e] = f;
  }
}

}  // namespace

extern "C" int fx_fill_normal(void* dst, int bf16, int64_t count, int64_t start, uint64_t key, double sd,
                              uint64_t nkey, double nsd, int noise, void* stream) {
  if (count <= 0) return 0;
  int64_t blocks = (count + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  fill_normal_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(dst, bf16, count, start, key, sd, nkey,
                                                                          nsd, noise);
  return (int)cudaGetLastError();
}
