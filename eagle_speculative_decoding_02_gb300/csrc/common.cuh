// Shared definitions of the EAGLE step kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace eg {

using bf16 = __nv_bfloat16;

// GEMM output tile width: weight rows per tile, and the column width of the
// per-row sum-of-squares partials that feed the next RMSNorm.
constexpr int kTileN = 128;
constexpr int kMaxTreeRows = 121;
constexpr int kMaxDepth = 8;
constexpr int kMaxTopK = 16;

// Device status word values (mirror eagle_status).
enum : int { kStOk = 0, kStInvalid = 1, kStCapacity = 4, kStTimeout = 6 };

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

// Store v as a GEMM input: hi[at] = T(v) and, when lo is given (bf16 models),
// lo[at] = bf16(v - hi), so that hi + lo carries v to about 16 mantissa bits.
template <typename T>
__device__ __forceinline__ void store_hilo(T* hi, bf16* lo, size_t at, float v) {
  const T h = from_f<T>(v);
  hi[at] = h;
  if (lo) lo[at] = __float2bfloat16_rn(v - to_f(h));
}

// store_hilo of four neighbouring elements (at a multiple of 4).
template <typename T>
__device__ __forceinline__ void store_hilo4(T* hi, bf16* lo, size_t at, float4 v) {
  if constexpr (sizeof(T) == 2) {
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y), h1 = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&h0);
    u.y = *reinterpret_cast<const uint32_t*>(&h1);
    *reinterpret_cast<uint2*>(hi + at) = u;
    if (lo) {
      const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
      const __nv_bfloat162 l0 = __floats2bfloat162_rn(v.x - f0.x, v.y - f0.y);
      const __nv_bfloat162 l1 = __floats2bfloat162_rn(v.z - f1.x, v.w - f1.y);
      uint2 w;
      w.x = *reinterpret_cast<const uint32_t*>(&l0);
      w.y = *reinterpret_cast<const uint32_t*>(&l1);
      *reinterpret_cast<uint2*>(lo + at) = w;
    }
  } else {
    store_hilo<T>(hi, lo, at, v.x);
    store_hilo<T>(hi, lo, at + 1, v.y);
    store_hilo<T>(hi, lo, at + 2, v.z);
    store_hilo<T>(hi, lo, at + 3, v.w);
  }
}

// KV-cache element type: the model dtype for float32 models; IEEE half for bf16
// models (11-bit significand, 8x finer than bf16, at the same two bytes; the
// attention products then run as f16 MMAs). Stores saturate at the half range;
// NaN passes through.
template <typename T> struct KvOf { using type = T; };
template <> struct KvOf<bf16> { using type = __half; };
template <typename T> __device__ __forceinline__ typename KvOf<T>::type kv_from_f(float v);
template <> __device__ __forceinline__ float kv_from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __half kv_from_f<bf16>(float v) {
  return __float2half_rn(v > 65504.f ? 65504.f : (v < -65504.f ? -65504.f : v));
}

__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, kStOk, code);
}

// Per-row metadata of one forward phase (verify, catch-up, draft depth, prefill chunk).
struct Rows {
  int* seq;        // [M] sequence index
  int* pos;        // [M] RoPE position
  int* slot;       // [M] KV slot to write, -1 = none (padding row)
  int* grp;        // [M] attention group
  uint64_t* mask;  // [M][2] visibility over the group's tree block
  int* tok;        // [M] input token (embedding row)
  int* fsrc;       // [M] feature row feeding the draft head's FC (draft phases)
};

// Rows of one sequence that share a fully visible prefix [0, prefix) and a
// tree block of slots [prefix, prefix + block_len) seen through per-row masks.
struct Group {
  int seq, row0, nrows, prefix, block_len;
};

enum EpiKind : int {
  kEpiStore = 0,   // y_f32[m][n] = acc * r_m
  kEpiQkv = 1,     // RoPE on q/k, q -> out (when set) and qg, k/v -> KV cache slots
  kEpiSwiglu = 2,  // silu(gate) * up over interleaved 64-row blocks -> out
  kEpiResid = 3,   // h += acc; hb = h * gain_next; per-tile sum of squares of h
  kEpiFc = 4,      // h = acc; hb = h * gain_next; per-tile sum of squares
  kEpiLmHead = 5,  // per-row top-k, max and sum-exp per vocab tile (+ optional logits)
};

struct EpiParams {
  int kind = kEpiStore;
  int M = 0, N = 0;
  // Row scale of RMSNorm applied after the product: r_m = 1/sqrt(sum_j ssq_in[j][m] / d_in + eps).
  const float* ssq_in = nullptr;
  int n_ssq_in = 0;
  float inv_d_in = 0.f;
  float eps = 0.f;
  float* y = nullptr;       // kEpiStore output; kEpiLmHead optional logits [M][N]
  void* out = nullptr;      // q (kEpiQkv, float32) [M][q_dim] or act (kEpiSwiglu, T) [M][ffn]
  // bf16 models carry GEMM inputs as hi/lo pairs (x = hi + lo): the low halves of
  // act (kEpiSwiglu) and hb (kEpiResid / kEpiFc); NULL for float32 models.
  bf16* out_lo = nullptr;
  bf16* hb_lo = nullptr;
  // kEpiQkv
  int q_dim = 0, kv_dim = 0, head_dim = 0, n_kv = 0, cap = 0;
  const float* rope_cos = nullptr;  // [positions][head_dim/2]
  const float* rope_sin = nullptr;
  void* kc = nullptr;       // layer cache base [B][n_kv][cap][head_dim], KvOf<T> elements
  void* vc = nullptr;
  Rows rows{};
  // optional: q again as half, times qg_scale, grouped by KV head,
  // [n_kv][M][q_dim / head_dim / n_kv][head_dim] (the query tiles of the
  // tensor-core attention: the GQA rows of one KV head are consecutive)
  __half* qg = nullptr;
  float qg_scale = 0.f;
  // kEpiSwiglu
  int ffn = 0;
  // kEpiResid / kEpiFc
  float* h = nullptr;       // [M][N] float32 residual stream
  void* hb = nullptr;       // [M][N] next GEMM input (h * gain_next)
  float* ssq_out = nullptr; // [N/128][M]
  const float* gain = nullptr;
  float* h_tap = nullptr;   // kEpiResid: optional copies of the new residual h (a feature tap of this layer)
  float* h_tap2 = nullptr;
  // kEpiLmHead
  int topk = 1;
  // sampling (inv_temp > 0): the top-k is taken of logit * inv_temp + Gumbel noise
  // (sample_gumbel) of (seq, position + 1, token) of each row; samp_pos / samp_seq
  // give a row's position and sequence, through samp_idx[row] when not NULL
  float inv_temp = 0.f;
  unsigned long long seed = 0;
  const int* samp_pos = nullptr;
  const int* samp_seq = nullptr;
  const int* samp_idx = nullptr;
  float* rec_val = nullptr; // [ntiles][M][topk]
  int* rec_idx = nullptr;
  float* rec_max = nullptr; // [ntiles][M]
  float* rec_sum = nullptr; // [ntiles][M] sum exp(logit - tile max)
};

// Programmatic dependent launch. A kernel launched with launch_pdl may start
// while its predecessor is still running; it must call pdl_wait() before it
// reads or writes anything the predecessor touches (every kernel here does so
// first thing), which makes ordering identical to a plain launch while the
// launch latency overlaps the predecessor's tail.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Barriers for code shared by whole-block and warp-specialised kernels.
struct BlockSync {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};
// Named barrier 1 over the 128 epilogue threads of a warp-specialised kernel.
struct EpilogueSync {
  __device__ __forceinline__ void operator()() const { asm volatile("bar.sync 1, 128;" ::: "memory"); }
};

__device__ __forceinline__ float silu_f(float x) { return x / (1.f + __expf(-x)); }

// SplitMix64's output function (Steele, Lea & Flood, OOPSLA 2014).
__device__ __forceinline__ unsigned long long mix64(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Gumbel noise of vocabulary entry v of the token at position pos of sequence
// seq: -log(-log(u)), u from a counter of (seed, seq, pos, v) (the definition
// in include/eagle.h). argmax over v of logit / T + noise samples softmax(logit / T).
__device__ __forceinline__ float sample_gumbel(unsigned long long seed, int seq, int pos, int v) {
  constexpr unsigned long long G = 0x9E3779B97F4A7C15ull;
  const unsigned long long k1 = mix64(seed + (unsigned long long)(seq + 1) * G);
  const unsigned long long k2 = mix64(k1 + (unsigned long long)(pos + 1) * G);
  const unsigned long long z = mix64(k2 + (unsigned long long)(v + 1) * G);
  const float u = ((float)(z >> 40) + 0.5f) * 5.9604644775390625e-08f;  // exact: (0, 1) on a 2^-24 grid
  return -logf(-logf(u));
}

// Warp arg-max on (value desc, index asc).
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace eg
