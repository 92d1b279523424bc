// Weight-only int4 projections: the library's block layout and the code-to-bf16
// conversion shared by the persistent kernel and the standalone dequantiser.
//
// "EAGLE (LLM decoding)", operational notes: EAGLE works with GPTQ / AWQ 4-bit
// weight-quantised targets. Format (symmetric, group-wise): a weight [N, K] is
// 4-bit codes u in [0, 15] and one bfloat16 scale s per row and group of 64
// inputs; W(n, k) = bf16(s(n, k / 64) * (u(n, k) - 8)), rounded once.
//
// Block layout (what the kernels stream): the weight is cut into blocks of
// 128 rows x 64 inputs, block (t, kb) at byte ((t * K/64) + kb) * kInt4BlockBytes.
// A block holds 128 rows of 8 code words (32 bytes per row), then the 128 rows'
// scales (bf16). Word c of a row carries inputs 8c .. 8c+7: input 8c + 2i in
// bits [4i, 4i+4) and input 8c + 2i + 1 in bits [16 + 4i, 20 + 4i), i = 0..3,
// so that (word >> 4i) & 0x000F000F puts two neighbouring inputs in the two
// halves of a bf16x2 register.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"

namespace eg {

constexpr int kInt4Group = 64;
constexpr int kInt4Rows = 128;
constexpr int kInt4CodeBytes = kInt4Rows * kInt4Group / 2;           // 4096
constexpr int kInt4BlockBytes = kInt4CodeBytes + kInt4Rows * 2;        // 4352 (a multiple of 16)

__host__ __device__ constexpr size_t int4_packed_bytes(int N, int K) {
  return (size_t)(N / kInt4Rows) * (K / kInt4Group) * kInt4BlockBytes;
}

// Eight weights of one code word as four bf16x2 (inputs 8c .. 8c+7 in order):
// 0x4300 | u is the bf16 of 128 + u, minus 136 is u - 8 exactly, and the product
// with the scale is rounded once to bf16.
__device__ __forceinline__ uint4 int4_dequant8(uint32_t w, __nv_bfloat162 s2) {
  const __nv_bfloat162 off = __floats2bfloat162_rn(136.f, 136.f);
  uint32_t r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t t = ((w >> (4 * i)) & 0x000F000Fu) | 0x43004300u;
    __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&t);
    v = __hmul2(__hsub2(v, off), s2);
    r[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

}  // namespace eg
