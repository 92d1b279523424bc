// Row-wise kernels: embedding gather, draft-head FC input, row gather and the
// LM-head top-k merge across vocab tiles.
#include "kernels.h"

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
__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(const float* __restrict__ rec_val,
                                                                   const int* __restrict__ rec_idx,
                                                                   const float* __restrict__ rec_max,
                                                                   const float* __restrict__ rec_sum, int ntiles,
                                                                   int M, int k, int* out_idx, float* out_val,
                                                                   float* out_lse) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red_m[kMergeWarps], red_s[kMergeWarps];
  __shared__ float sv[kMergeWarps];
  __shared__ int si[kMergeWarps];
  const int m = blockIdx.x, tid = threadIdx.x;
  // (max, sum of exp(x - max)) pairs: combining keeps the larger max
  auto combine = [](float& am, float& as, float bm, float bs) {
    if (bm == -INFINITY) return;
    if (am == -INFINITY) {
      am = bm;
      as = bs;
    } else if (bm > am) {
      as = as * __expf(am - bm) + bs;
      am = bm;
    } else {
      as += bs * __expf(bm - am);
    }
  };
  float rm = -INFINITY, rs = 0.f;
  // Each thread keeps the k best of its candidates (value desc, index asc), sorted, in registers.
  float lv[kMaxTopK];
  int li[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    lv[j] = -INFINITY;
    li[j] = 0x7fffffff;
  }
  constexpr int kU = 2;
  for (int t0 = tid; t0 < ntiles; t0 += kU * kMergeThreads) {
    float tm[kU], ts[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int t = t0 + u * kMergeThreads;
      const size_t r = (size_t)t * M + m;
      tm[u] = t < ntiles ? rec_max[r] : -INFINITY;
      ts[u] = t < ntiles ? rec_sum[r] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) combine(rm, rs, tm[u], ts[u]);
    for (int u = 0; u < kU; ++u) {
      const int t = t0 + u * kMergeThreads;
      if (t >= ntiles) break;
      // the tile's best is its max: nothing of the tile enters unless that does
      if (!(tm[u] >= lv[k - 1])) continue;
      const size_t base = ((size_t)t * M + m) * k;
      float cv[kMaxTopK];
      int cx[kMaxTopK];
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {  // the tile's candidates, all loads in flight
        cv[j] = j < k ? rec_val[base + j] : -INFINITY;
        cx[j] = j < k ? rec_idx[base + j] : -1;
      }
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {
        // candidates of one tile arrive sorted: once one misses the list, the rest of the tile does too
        if (j >= k || cx[j] < 0 || !(cv[j] > lv[k - 1] || (cv[j] == lv[k - 1] && cx[j] < li[k - 1]))) break;
        float c = cv[j];
        int ci = cx[j];
#pragma unroll
        for (int q = 0; q < kMaxTopK; ++q) {
          if (q < k && (c > lv[q] || (c == lv[q] && ci < li[q]))) {
            const float tv = lv[q];
            const int ti = li[q];
            lv[q] = c;
            li[q] = ci;
            c = tv;
            ci = ti;
          }
        }
      }
    }
  }
  // (max, sum) over the block: warps by shuffles, then the warps in order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, rm, o), os = __shfl_xor_sync(0xffffffffu, rs, o);
    combine(rm, rs, om, os);
  }
  if ((tid & 31) == 0) {
    red_m[tid >> 5] = rm;
    red_s[tid >> 5] = rs;
  }
  __syncthreads();
  if (tid == 0 && out_lse) {
    float gm = red_m[0], gs = red_s[0];
    for (int w = 1; w < kMergeWarps; ++w) combine(gm, gs, red_m[w], red_s[w]);
    out_lse[m] = gm + __logf(gs);
  }

  // k rounds of a block arg-max over the heads of the sorted lists
  int head = 0;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int q = 0; q < kMaxTopK; ++q)
      if (q == head) {
        bv = lv[q];
        bi = li[q];
      }
    const int mine = bi;
    warp_argmax(bv, bi);
    __syncthreads();
    if ((tid & 31) == 0) {
      sv[tid >> 5] = bv;
      si[tid >> 5] = bi;
    }
    __syncthreads();
    bv = sv[0];
    bi = si[0];
    for (int w = 1; w < kMergeWarps; ++w)
      if (sv[w] > bv || (sv[w] == bv && si[w] < bi)) {
        bv = sv[w];
        bi = si[w];
      }
    if (mine == bi && head < k) ++head;  // indices are unique: exactly one list owns the winner
    if (tid == 0) {
      out_idx[(size_t)m * k + r] = bi == 0x7fffffff ? -1 : bi;
      if (out_val) out_val[(size_t)m * k + r] = bv;
    }
  }
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
  return launch_pdl(topk_merge_kernel, dim3(M), dim3(kMergeThreads), 0, s, rec_val, rec_idx, rec_max, rec_sum, ntiles, M, k, idx, val, lse);
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
