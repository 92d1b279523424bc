// Device-side implementation of the fixture generator defined in
// fixtures/__init__.py (SplitMix64 words, Box-Muller normals in float64,
// rounded to float32 and then to bfloat16). Fills the 8B / 70B-shaped weights
// in place on the GPU; the oracle draws the same numbers with numpy.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

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

// Byte (n, i) of a packed int4 projection [N, K]: codes (n, 2i) and (n, 2i+1),
// each 1 + ((word(key, n K + k) >> 32) * 15 >> 32).
__global__ void fill_int4_codes_kernel(uint8_t* dst, int64_t n_bytes, uint64_t key) {
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n_bytes;
       e += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t j = 2 * (uint64_t)e;  // element index n K + 2i (K is even)
    const uint64_t w0 = mix64(key + (j + 1) * kGamma), w1 = mix64(key + (j + 2) * kGamma);
    const uint32_t c0 = 1u + (uint32_t)(((w0 >> 32) * 15ull) >> 32);
    const uint32_t c1 = 1u + (uint32_t)(((w1 >> 32) * 15ull) >> 32);
    dst[e] = (uint8_t)(c0 | (c1 << 4));
  }
}

// Group scale g: bf16(float(b (0.75 + 0.5 r))), r = (word(key, g) >> 11) 2^-53.
__global__ void fill_int4_scales_kernel(__nv_bfloat16* dst, int64_t count, uint64_t key, double b) {
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < count;
       e += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t w = mix64(key + ((uint64_t)e + 1) * kGamma);
    const double r = (double)(w >> 11) * (1.0 / 9007199254740992.0);
    dst[e] = __float2bfloat16_rn((float)(b * (0.75 + 0.5 * r)));
  }
}

}  // namespace

extern "C" int fx_fill_int4(void* codes, void* scales, int64_t n, int64_t k, uint64_t key_codes,
                            uint64_t key_scales, double base, void* stream) {
  if (n <= 0 || k <= 0 || (k % 64)) return 1;
  const cudaStream_t s = (cudaStream_t)stream;
  const int64_t nb = n * k / 2, ng = n * (k / 64);
  fill_int4_codes_kernel<<<(unsigned)std::min<int64_t>((nb + 255) / 256, 152 * 64), 256, 0, s>>>(
      (uint8_t*)codes, nb, key_codes);
  fill_int4_scales_kernel<<<(unsigned)std::min<int64_t>((ng + 255) / 256, 152 * 64), 256, 0, s>>>(
      (__nv_bfloat16*)scales, ng, key_scales, base);
  return (int)cudaGetLastError();
}

extern "C" int fx_fill_normal(void* dst, int bf16, int64_t count, int64_t start, uint64_t key, double sd,
                              uint64_t nkey, double nsd, int noise, void* stream) {
  if (count <= 0) return 0;
  int64_t blocks = (count + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  fill_normal_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(dst, bf16, count, start, key, sd, nkey,
                                                                          nsd, noise);
  return (int)cudaGetLastError();
}
