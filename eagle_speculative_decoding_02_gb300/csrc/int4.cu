// Weight-only int4: repacking plain codes into the library's block layout, and
// expanding blocks to dense weights for the per-operation GEMMs (prefill, wide
// verify batches, float32 models). The persistent kernel expands the blocks in
// shared memory instead (stack_tc.cu). Format and layout: int4.cuh.
#include "../../include/eagle.h"
#include "int4.cuh"
#include "kernels.h"

namespace eg {
namespace {

// One thread per (row, 64-input group, code word): word c of row n in block
// (n / 128, g) from the plain bytes 32 g + 4c .. 32 g + 4c + 3 of the row (byte
// b holds inputs 2b and 2b + 1 in its low and high nibble); the c = 0 thread
// also copies the scale.
__global__ void int4_pack_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales, int N,
                                 int K, uint8_t* __restrict__ out) {
  const int G = K / kInt4Group;
  const long long total = (long long)N * G * 8;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(e & 7);
    const long long ng = e >> 3;
    const int n = (int)(ng / G), g = (int)(ng % G);
    const uint8_t* src = codes + (size_t)n * (K / 2) + (size_t)g * 32 + 4 * c;
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t b = src[i];
      w |= (b & 0xFu) << (4 * i);          // input 8c + 2i
      w |= (b >> 4) << (16 + 4 * i);       // input 8c + 2i + 1
    }
    uint8_t* blk = out + ((size_t)(n / kInt4Rows) * G + g) * kInt4BlockBytes;
    const int r = n % kInt4Rows;
    reinterpret_cast<uint32_t*>(blk + (size_t)r * 32)[c] = w;
    if (c == 0) reinterpret_cast<uint16_t*>(blk + kInt4CodeBytes)[r] = scales[(size_t)n * G + g];
  }
}

// Dense weights [N][K] from blocks: one thread per (row, group, word), 8 outputs.
template <typename T>
__global__ void int4_dequant_kernel(const uint8_t* __restrict__ w4, int N, int K, T* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int G = K / kInt4Group;
  const long long total = (long long)N * G * 8;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(e & 7);
    const long long ng = e >> 3;
    const int n = (int)(ng / G), g = (int)(ng % G);
    const uint8_t* blk = w4 + ((size_t)(n / kInt4Rows) * G + g) * kInt4BlockBytes;
    const int r = n % kInt4Rows;
    const uint32_t w = reinterpret_cast<const uint32_t*>(blk + (size_t)r * 32)[c];
    const __nv_bfloat16 s = reinterpret_cast<const __nv_bfloat16*>(blk + kInt4CodeBytes)[r];
    const uint4 v = int4_dequant8(w, __halves2bfloat162(s, s));
    T* dst = out + (size_t)n * K + (size_t)g * kInt4Group + 8 * c;
    if constexpr (sizeof(T) == 2) {
      *reinterpret_cast<uint4*>(dst) = v;
    } else {
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(&u[i]);
        dst[2 * i] = __bfloat162float(p.x);
        dst[2 * i + 1] = __bfloat162float(p.y);
      }
    }
  }
}

unsigned grid_for(long long n) {
  long long b = (n + 255) / 256;
  return (unsigned)(b < 1 ? 1 : (b > 152 * 16 ? 152 * 16 : b));
}

}  // namespace

bool int4_shape_ok(int N, int K) { return N > 0 && K > 0 && N % kInt4Rows == 0 && K % kInt4Group == 0; }

template <typename T>
cudaError_t int4_dequant(const void* w4, int N, int K, T* out, cudaStream_t s) {
  if (!int4_shape_ok(N, K)) return cudaErrorInvalidValue;
  return launch_pdl(int4_dequant_kernel<T>, dim3(grid_for((long long)N * (K / kInt4Group) * 8)), dim3(256), 0, s,
                    (const uint8_t*)w4, N, K, out);
}
template cudaError_t int4_dequant<float>(const void*, int, int, float*, cudaStream_t);
template cudaError_t int4_dequant<bf16>(const void*, int, int, bf16*, cudaStream_t);

}  // namespace eg

extern "C" {

size_t eagle_int4_packed_bytes(int32_t N, int32_t K) {
  return eg::int4_shape_ok(N, K) ? eg::int4_packed_bytes(N, K) : 0;
}

eagle_status eagle_int4_pack(const uint8_t* d_codes, const uint16_t* d_scales, int32_t N, int32_t K, void* d_out,
                             void* stream) {
  using namespace eg;
  if (!d_codes || !d_scales || !d_out) return EAGLE_ERR_INVALID_ARG;
  if (!int4_shape_ok(N, K)) return EAGLE_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(d_out) & 15) != 0) return EAGLE_ERR_INVALID_ARG;
  int4_pack_kernel<<<grid_for((long long)N * (K / kInt4Group) * 8), 256, 0, (cudaStream_t)stream>>>(
      d_codes, d_scales, N, K, (uint8_t*)d_out);
  return cudaGetLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

eagle_status eagle_op_int4_dequant(const void* d_w4, int32_t N, int32_t K, int32_t dtype, void* d_out,
                                   void* stream) {
  using namespace eg;
  if (!d_w4 || !d_out) return EAGLE_ERR_INVALID_ARG;
  if (!int4_shape_ok(N, K)) return EAGLE_ERR_UNSUPPORTED;
  cudaError_t e;
  if (dtype == EAGLE_DTYPE_F32)
    e = int4_dequant<float>(d_w4, N, K, (float*)d_out, (cudaStream_t)stream);
  else if (dtype == EAGLE_DTYPE_BF16)
    e = int4_dequant<bf16>(d_w4, N, K, (bf16*)d_out, (cudaStream_t)stream);
  else
    return EAGLE_ERR_INVALID_ARG;
  return e == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

}  // extern "C"
