// Host-side launchers of the EAGLE step kernels.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace eg {

// ---- GEMM: Y = X W^T with a fused epilogue ------------------------------------------------------
template <typename T>
cudaError_t gemm_simt(const T* X, const T* W, int M, int N, int K, const EpiParams& ep, cudaStream_t s);

// tcgen05 + TMA weight-streaming GEMM (bf16). `scratch` holds split-K partials
// and per-tile arrival counters (counters must start at zero; the kernel
// leaves them at zero). Returns cudaErrorInvalidValue for unsupported shapes.
// X_lo (may be NULL): low halves of a hi/lo activation pair, Y = (X + X_lo) W^T.
size_t gemm_tc_scratch_bytes(int M, int N, int K);
// w_dep: W was written by the previous kernel on the stream (for example an
// expanded int4 weight); otherwise the weight boxes of the first stages are
// requested before the programmatic-dependent-launch wait.
cudaError_t gemm_tc(const bf16* X, const bf16* X_lo, const bf16* W, int M, int N, int K, const EpiParams& ep,
                    void* scratch, int* status, cudaStream_t s, bool w_dep = false);

// 2D bf16 tensor map of a row-major [rows][cols] matrix, box [box_rows][64],
// 128-byte swizzle (the operand format of the tcgen05 kernels).
bool make_tmap_bf16(CUtensorMap* m, const void* base, int rows, int cols, int box_rows);
// The same for IEEE half elements (the KV cache of bf16 models).
bool make_tmap_f16(CUtensorMap* m, const void* base, int rows, int cols, int box_rows);
// SMs of the current device (capped at the scratch-sizing bound).
int num_sms();
// Raise a kernel's dynamic shared-memory limit on the current device (once per device).
bool raise_smem_limit(const void* kernel, int bytes);

// ---- weight-only int4 (int4.cuh: format and block layout) --------------------------------------
bool int4_shape_ok(int N, int K);
// Dense [N][K] weights of T from a packed int4 weight (the per-operation GEMMs' input).
template <typename T>
cudaError_t int4_dequant(const void* w4, int N, int K, T* out, cudaStream_t s);

// ---- attention ---------------------------------------------------------------------------------
struct AttnArgs {
  const float* q;     // [M][Hq][hd] float32 (RoPE applied)
  const __half* qg;   // optional: q * scale * log2(e) as half, [Hkv][M][Hq / Hkv][hd]
  const void* kc;     // [B][Hkv][cap][hd]
  const void* vc;
  void* o;            // [M][Hq * hd]
  bf16* o_lo;         // low halves of o as a hi/lo pair (bf16 models; may be NULL)
  const Group* groups;
  int n_groups;
  const uint64_t* mask;  // [M][2]
  const int* row_grp;    // [M] group of each row (NULL: all rows in group 0)
  int M, Hq, Hkv, hd, cap;
  int n_seq;          // sequences the cache holds: kc / vc have n_seq * Hkv * cap rows
  int max_prefix;     // upper bound on any group's prefix (sizes the split grid)
  float scale;        // 1/sqrt(hd)
  float* part;        // split partials (tensor-core path)
  int* status;
};
template <typename T>
cudaError_t attention_simt(const AttnArgs& a, cudaStream_t s);
// The tcgen05 tree attention (bf16 models: half KV cache) as two launches
// (items, then merge) of the persistent kernel's attention code; needs
// a.qg and a.part of attention_umma_part_bytes(M, Hq, Hkv, hd, max_prefix) bytes.
size_t attention_umma_part_bytes(int M, int Hq, int Hkv, int hd, int max_prefix);
cudaError_t attention_umma(const AttnArgs& a, cudaStream_t s);
// The grouped half queries a.qg from float32 queries q [M][Hq][hd].
cudaError_t attention_umma_qg(const float* q, int M, int Hq, int Hkv, int hd, float scale, __half* qg,
                              cudaStream_t s);

// ---- rows, embeddings, FC input ----------------------------------------------------------------
template <typename T>
cudaError_t embed_rows(const T* E, const int* tok, int M, int d, const float* gain, float* h, T* hb, bf16* hb_lo,
                       float* ssq, cudaStream_t s);
template <typename T>
cudaError_t fc_input(const float* feat, const int* fsrc, const T* E, const int* tok, int M, int d, T* x, bf16* x_lo,
                     cudaStream_t s);
// x[m] = [low[m] ; mid[m] ; top[m]] for m < M (3d wide; hi/lo pair when x_lo is given).
template <typename T>
cudaError_t pack_taps(const float* low, const float* mid, const float* top, int M, int d, T* x, bf16* x_lo,
                      cudaStream_t s);
// Copy rows src[i] of (hb, hb_lo, ssq) to rows i of (hb_dst, lo_dst, ssq_dst); the lo pointers may be NULL.
template <typename T>
cudaError_t gather_rows(const T* hb, const bf16* hb_lo, const float* ssq, int M_src, const int* src, int n, int d,
                        T* hb_dst, bf16* lo_dst, float* ssq_dst, cudaStream_t s);

// ---- LM-head top-k merge over vocab tiles ------------------------------------------------------
cudaError_t topk_merge(const float* rec_val, const int* rec_idx, const float* rec_max, const float* rec_sum,
                       int ntiles, int M, int k, int* idx, float* val, float* lse, cudaStream_t s);

}  // namespace eg
