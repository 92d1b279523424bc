// Row-wise kernels: embedding gather, draft-head FC input, row gather and the
// LM-head top-k merge across vocab tiles.
#include "kernels.h"
#include "topk.cuh"

namespace eg {
namespace {

// Block sum over 128 threads in a fixed order (warp tree, then warps 0..3).
__device__ float block_sum128(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  return ((red[0] + red[1]) + red[2]) + red[3];
}

// h = E[tok]; hb (+ hb_lo) = h * gain; ssq[j][m] = sum of h^2 over column tile j.
template <typename T>
__global__ void __launch_bounds__(128) embed_kernel(const T* __restrict__ E, const int* __restrict__ tok, int M,
                                                    int d, const float* __restrict__ gain, float* h, T* hb,
                                                    bf16* hb_lo, float* ssq) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[4];
  const int m = blockIdx.x;
  const int t = tok[m];
  for (int j = 0; j * kTileN < d; ++j) {
    const int n = j * kTileN + threadIdx.x;
    float v = 0.f;
    if (n < d) {
      v = to_f(E[(size_t)t * d + n]);
      h[(size_t)m * d + n] = v;
      store_hilo<T>(hb, hb_lo, (size_t)m * d + n, v * gain[n]);
    }
    const float s = block_sum128(v * v, red);
    if (threadIdx.x == 0) ssq[(size_t)j * M + m] = s;
  }
}

// Input rows of the fused-feature matrix: x[m] = [low[m] ; mid[m] ; top[m]] (3d
// wide), as a hi/lo pair for bf16 models.
template <typename T>
__global__ void pack_taps_kernel(const float* __restrict__ low, const float* __restrict__ mid,
                                 const float* __restrict__ top, int d, T* x, bf16* x_lo) {
  pdl_wait();
  pdl_trigger();
  const size_t m = blockIdx.x;
  const size_t row = m * 3 * d;
  for (int n = threadIdx.x; n < d; n += blockDim.x) {
    store_hilo<T>(x, x_lo, row + n, low[m * d + n]);
    store_hilo<T>(x, x_lo, row + d + n, mid[m * d + n]);
    store_hilo<T>(x, x_lo, row + 2 * d + n, top[m * d + n]);
  }
}

// x[m] = [ feat[fsrc[m]] ; E[tok[m]] ] (length 2d); the float feature half is
// stored as a hi/lo pair when x_lo is given, the embedding half is exact.
template <typename T>
__global__ void fc_input_kernel(const float* __restrict__ feat, const int* __restrict__ fsrc,
                                const T* __restrict__ E, const int* __restrict__ tok, int d, T* x, bf16* x_lo) {
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.x;
  const float* f = feat + (size_t)fsrc[m] * d;
  const T* e = E + (size_t)tok[m] * d;
  const size_t row = (size_t)m * 2 * d;
#pragma unroll 4
  for (int n = threadIdx.x; n < d; n += blockDim.x) {
    store_hilo<T>(x, x_lo, row + n, f[n]);
    x[row + d + n] = e[n];
    if (x_lo) x_lo[row + d + n] = __float2bfloat16_rn(0.f);
  }
}

template <typename T>
__global__ void gather_rows_kernel(const T* __restrict__ hb, const bf16* __restrict__ hb_lo,
                                   const float* __restrict__ ssq, int M_src, const int* __restrict__ src, int n_rows,
                                   int d, T* hb_dst, bf16* lo_dst, float* ssq_dst) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  const int r = src[i];
  for (int n = threadIdx.x; n < d; n += blockDim.x) {
    hb_dst[(size_t)i * d + n] = hb[(size_t)r * d + n];
    if (lo_dst) lo_dst[(size_t)i * d + n] = hb_lo[(size_t)r * d + n];
  }
  for (int j = threadIdx.x; j * kTileN < d; j += blockDim.x) ssq_dst[(size_t)j * n_rows + i] = ssq[(size_t)j * M_src + r];
}

// One block per row: log-sum-exp over all vocab tiles and the k best (value desc,
// index asc) of the per-tile candidates, in one pass over the row's records:
// each thread takes tiles tid, tid + 512, ... (all their loads in flight), keeps a
// running (max, sum of exp(x - max)) and its own sorted k best; the block then
// combines the pairs in fixed order and merges the lists.
constexpr int kMergeThreads = 512;
constexpr int kMergeWarps = kMergeThreads / 32;
__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(TopkMerge g) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[4 * kMergeWarps];
  struct Sync {
    __device__ void operator()() const { __syncthreads(); }
  };
  topk_merge_row<kMergeThreads>(g, blockIdx.x, threadIdx.x, red, Sync{});
}

}  // namespace

template <typename T>
cudaError_t embed_rows(const T* E, const int* tok, int M, int d, const float* gain, float* h, T* hb, bf16* hb_lo,
                       float* ssq, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  return launch_pdl(embed_kernel<T>, dim3(M), dim3(128), 0, s, E, tok, M, d, gain, h, hb, hb_lo, ssq);
}

template <typename T>
cudaError_t fc_input(const float* feat, const int* fsrc, const T* E, const int* tok, int M, int d, T* x, bf16* x_lo,
                     cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  return launch_pdl(fc_input_kernel<T>, dim3(M), dim3(256), 0, s, feat, fsrc, E, tok, d, x, x_lo);
}

template <typename T>
cudaError_t pack_taps(const float* low, const float* mid, const float* top, int M, int d, T* x, bf16* x_lo,
                      cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  return launch_pdl(pack_taps_kernel<T>, dim3(M), dim3(256), 0, s, low, mid, top, d, x, x_lo);
}

template <typename T>
cudaError_t gather_rows(const T* hb, const bf16* hb_lo, const float* ssq, int M_src, const int* src, int n, int d,
                        T* hb_dst, bf16* lo_dst, float* ssq_dst, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(gather_rows_kernel<T>, dim3(n), dim3(256), 0, s, hb, hb_lo, ssq, M_src, src, n, d, hb_dst, lo_dst, ssq_dst);
}

cudaError_t topk_merge(const float* rec_val, const int* rec_idx, const float* rec_max, const float* rec_sum,
                       int ntiles, int M, int k, int* idx, float* val, float* lse, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  TopkMerge g;
  g.val = rec_val;
  g.idx = rec_idx;
  g.mx = rec_max;
  g.sum = rec_sum;
  g.ntiles = ntiles;
  g.M = M;
  g.k = k;
  g.out_idx = idx;
  g.out_val = val;
  g.out_lse = lse;
  return launch_pdl(topk_merge_kernel, dim3(M), dim3(kMergeThreads), 0, s, g);
}

#define EG_INST(T)                                                                                          \
  template cudaError_t embed_rows<T>(const T*, const int*, int, int, const float*, float*, T*, bf16*, float*,  \
                                     cudaStream_t);                                                         \
  template cudaError_t fc_input<T>(const float*, const int*, const T*, const int*, int, int, T*, bf16*,      \
                                   cudaStream_t);                                                           \
  template cudaError_t pack_taps<T>(const float*, const float*, const float*, int, int, T*, bf16*, cudaStream_t); \
  template cudaError_t gather_rows<T>(const T*, const bf16*, const float*, int, const int*, int, int, T*, bf16*, \
                                      float*, cudaStream_t);
EG_INST(float)
EG_INST(bf16)
#undef EG_INST

}  // namespace eg
