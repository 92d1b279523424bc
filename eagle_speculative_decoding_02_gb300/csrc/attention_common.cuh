// Helpers shared by the tree-attention code: the layout of the split partials
// and small conversions.
#pragma once

#include <cmath>

#include "kernels.h"

namespace eg {
namespace attn {

__device__ __forceinline__ uint32_t pack_half2(float x, float y) {
  const __half2 h = __floats2half2_rn(x, y);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__host__ __device__ __forceinline__ int n_prefix_chunks(int prefix, int ck) { return (prefix + ck - 1) / ck; }

// Split partials of chunk slot c (of `slots`) and pair w = row * Hq + query head
// (of Mw = M * Hq): the unnormalised output in HD / 32 blocks of 32 columns,
// [slots][HD / 32][Mw][32] (a row's block is 128 contiguous bytes), then the
// (max, sum) pairs [slots][Mw][2]; slots * Mw * (HD + 2) floats in all.
struct PartLayout {
  float* base;
  int Mw, slots, hd;
  __device__ float* o(int c, int w, int blk) const { return base + (((size_t)c * (hd / 32) + blk) * Mw + w) * 32; }
  __device__ float* ml(int c, int w) const { return base + (size_t)slots * hd * Mw + ((size_t)c * Mw + w) * 2; }
};

}  // namespace attn
}  // namespace eg
