// SIMT GEMM Y = X W^T with the shared epilogues: the float32 path (tiny
// correctness model, where tensor-core tf32 would miss the 1e-4 logit bound).
// Each output element is summed over k in ascending order, independent of M.
#include "epilogue.cuh"
#include "kernels.h"

namespace eg {

namespace {
constexpr int BM = 32, BK = 32, LDT = kTileN + 1;

template <typename T>
__global__ void __launch_bounds__(128) gemm_simt_kernel(const T* __restrict__ X, const T* __restrict__ W, int M,
                                                        int N, int K, EpiParams ep) {
  __shared__ float ws[BK][kTileN + 4];
  __shared__ float xs[BK][BM + 1];
  __shared__ float tile[BM * LDT];
  __shared__ float rscale[kEpiRowSmemFloats];
  const int tid = threadIdx.x;
  const int n0 = blockIdx.x * kTileN, m0 = blockIdx.y * BM;
  const int tn = tid & 31, tm = tid >> 5;  // thread computes cols tn+32i, rows tm*8+j
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += BK) {
    for (int e = tid; e < kTileN * BK; e += 128) {
      const int r = e / BK, kk = e % BK;
      const int n = n0 + r, k = k0 + kk;
      ws[kk][r] = (n < N && k < K) ? to_f(W[(size_t)n * K + k]) : 0.f;
    }
    for (int e = tid; e < BM * BK; e += 128) {
      const int r = e / BK, kk = e % BK;
      const int m = m0 + r, k = k0 + kk;
      xs[kk][r] = (m < M && k < K) ? to_f(X[(size_t)m * K + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < BK; ++kk) {
      float w[4], x[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = ws[kk][tn + 32 * i];
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = xs[kk][tm * 8 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(w[i], x[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) tile[(tm * 8 + j) * LDT + tn + 32 * i] = acc[i][j];
  __syncthreads();
  run_epilogue<T>(ep, tile, LDT, m0, min(BM, M - m0), n0, rscale, tid, BlockSync{});
}
}  // namespace

template <typename T>
cudaError_t gemm_simt(const T* X, const T* W, int M, int N, int K, const EpiParams& ep, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  dim3 grid((N + kTileN - 1) / kTileN, (M + BM - 1) / BM);
  gemm_simt_kernel<T><<<grid, 128, 0, s>>>(X, W, M, N, K, ep);
  return cudaGetLastError();
}

template cudaError_t gemm_simt<float>(const float*, const float*, int, int, int, const EpiParams&, cudaStream_t);
template cudaError_t gemm_simt<bf16>(const bf16*, const bf16*, int, int, int, const EpiParams&, cudaStream_t);

}  // namespace eg
