// Kernel-level C entry points (eagle_op_*): one hot-path kernel on caller
// buffers, for unit parity tests and roofline timing.
#include <cmath>

#include "../../include/eagle.h"
#include "kernels.h"

using namespace eg;

namespace {

size_t al(size_t v) { return (v + 255) / 256 * 256; }

__global__ void write_group_kernel(Group* g, int rows, int prefix, int block_len) {
  g->seq = 0;
  g->row0 = 0;
  g->nrows = rows;
  g->prefix = prefix;
  g->block_len = block_len;
}

}  // namespace

extern "C" {

size_t eagle_op_gemm_scratch_bytes(int32_t M, int32_t N, int32_t K, int32_t dtype) {
  if (dtype == EAGLE_DTYPE_BF16) return al(gemm_tc_scratch_bytes(M, N, K));
  return 256;
}

eagle_status eagle_op_gemm(int32_t dtype, int32_t M, int32_t N, int32_t K, const void* x, const void* x_lo,
                           const void* w, float* y, void* scratch, size_t scratch_bytes, void* stream) {
  if (M < 1 || N < 1 || K < 1 || !x || !w || !y) return EAGLE_ERR_INVALID_ARG;
  if (scratch_bytes < eagle_op_gemm_scratch_bytes(M, N, K, dtype)) return EAGLE_ERR_WORKSPACE;
  EpiParams e;
  e.kind = kEpiStore;
  e.M = M;
  e.N = N;
  e.y = y;
  cudaError_t err;
  if (dtype == EAGLE_DTYPE_BF16) {
    if (N % kTileN || K % 64) return EAGLE_ERR_UNSUPPORTED;
    if (!scratch) return EAGLE_ERR_WORKSPACE;
    err = gemm_tc((const bf16*)x, (const bf16*)x_lo, (const bf16*)w, M, N, K, e, scratch, nullptr,
                  (cudaStream_t)stream);
  } else if (dtype == EAGLE_DTYPE_F32) {
    err = gemm_simt<float>((const float*)x, (const float*)w, M, N, K, e, (cudaStream_t)stream);
  } else {
    return EAGLE_ERR_INVALID_ARG;
  }
  return err == cudaSuccess ? EAGLE_OK : (err == cudaErrorInvalidValue ? EAGLE_ERR_UNSUPPORTED : EAGLE_ERR_CUDA);
}

size_t eagle_op_lmhead_scratch_bytes(int32_t M, int32_t N, int32_t K, int32_t k, int32_t dtype) {
  const size_t nt = (size_t)((N + kTileN - 1) / kTileN) * M;
  size_t s = al(nt * k * 4) * 2 + al(nt * 4) * 2;
  if (dtype == EAGLE_DTYPE_BF16) s += al(gemm_tc_scratch_bytes(M, N, K));
  return s;
}

eagle_status eagle_op_lmhead_topk(int32_t dtype, int32_t M, int32_t N, int32_t K, int32_t k, const void* x,
                                  const void* w, int32_t* idx, float* val, float* lse, void* scratch,
                                  size_t scratch_bytes, void* stream) {
  if (M < 1 || N < 1 || K < 1 || k < 1 || k > EAGLE_MAX_TOPK || k > N || !x || !w || !idx || !scratch)
    return EAGLE_ERR_INVALID_ARG;
  if (scratch_bytes < eagle_op_lmhead_scratch_bytes(M, N, K, k, dtype)) return EAGLE_ERR_WORKSPACE;
  const size_t nt = (size_t)((N + kTileN - 1) / kTileN) * M;
  char* p = (char*)scratch;
  EpiParams e;
  e.kind = kEpiLmHead;
  e.M = M;
  e.N = N;
  e.topk = k;
  e.rec_val = (float*)p; p += al(nt * k * 4);
  e.rec_idx = (int*)p; p += al(nt * k * 4);
  e.rec_max = (float*)p; p += al(nt * 4);
  e.rec_sum = (float*)p; p += al(nt * 4);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t err;
  if (dtype == EAGLE_DTYPE_BF16) {
    if (N % kTileN || K % 64) return EAGLE_ERR_UNSUPPORTED;
    err = gemm_tc((const bf16*)x, nullptr, (const bf16*)w, M, N, K, e, p, nullptr, s);
  } else if (dtype == EAGLE_DTYPE_F32) {
    err = gemm_simt<float>((const float*)x, (const float*)w, M, N, K, e, s);
  } else {
    return EAGLE_ERR_INVALID_ARG;
  }
  if (err == cudaSuccess)
    err = topk_merge(e.rec_val, e.rec_idx, e.rec_max, e.rec_sum, (N + kTileN - 1) / kTileN, M, k, idx, val, lse, s);
  return err == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

size_t eagle_op_attention_scratch_bytes(int32_t rows, int32_t n_heads, int32_t hd, int32_t prefix) {
  // the group, then the partials (the larger of the two layouts), then the grouped half queries
  const size_t part = attention_umma_part_bytes(rows, n_heads, 1, hd, prefix + 128);
  return al(sizeof(Group)) + al(part) + al((size_t)rows * n_heads * hd * 2);
}

eagle_status eagle_op_tree_attention(int32_t dtype, int32_t rows, int32_t n_heads, int32_t n_kv_heads, int32_t hd,
                                     int32_t cap, int32_t prefix, const void* q, const void* k, const void* v,
                                     const uint64_t* mask, void* o, void* scratch, size_t scratch_bytes,
                                     void* stream) {
  if (rows < 1 || rows > 128 || n_heads < 1 || n_kv_heads < 1 || n_heads % n_kv_heads || (hd != 64 && hd != 128) ||
      prefix < 0 || prefix + rows > cap || !q || !k || !v || !mask || !o || !scratch)
    return EAGLE_ERR_INVALID_ARG;
  if (scratch_bytes < eagle_op_attention_scratch_bytes(rows, n_heads, hd, prefix)) return EAGLE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  Group* g = (Group*)scratch;
  write_group_kernel<<<1, 1, 0, s>>>(g, rows, prefix, rows);
  AttnArgs a{};
  a.q = (const float*)q; a.o_lo = nullptr; a.kc = k; a.vc = v; a.o = o; a.groups = g; a.n_groups = 1; a.mask = mask; a.row_grp = nullptr; a.M = rows;
  a.Hq = n_heads; a.Hkv = n_kv_heads; a.hd = hd; a.cap = cap; a.max_prefix = prefix;
  a.scale = 1.f / std::sqrt((float)hd);
  a.part = (float*)((char*)scratch + al(sizeof(Group)));
  a.status = nullptr;
  cudaError_t err;
  if (dtype == EAGLE_DTYPE_BF16) {
    // the tcgen05 items and merge, on grouped half queries made from q
    const size_t part = attention_umma_part_bytes(rows, n_heads, 1, hd, prefix + 128);
    __half* qg = (__half*)((char*)scratch + al(sizeof(Group)) + al(part));
    a.qg = qg;
    a.n_seq = 1;
    err = attention_umma_qg((const float*)q, rows, n_heads, n_kv_heads, hd, a.scale, qg, s);
    if (err == cudaSuccess) err = attention_umma(a, s);
  }
  else if (dtype == EAGLE_DTYPE_F32) err = attention_simt<float>(a, s);
  else return EAGLE_ERR_INVALID_ARG;
  return err == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}

}  // extern "C"
