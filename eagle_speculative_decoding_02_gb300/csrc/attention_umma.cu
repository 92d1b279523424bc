// Tree attention on the tcgen05 tensor cores as standalone launches: the
// persistent kernel's attention items and merge (attention_umma.cuh), each
// spread over one CTA per SM. Used where the persistent kernel does not run the
// pass: prefill chunks, verify passes of more rows than two persistent launches
// take, and the kernel-level ABI. ("EAGLE (LLM decoding)", section "How EAGLE
// works": every tree node attends to the committed prefix and to its ancestors
// in the tree block, in one pass.)
//
// Launch 1 (items): item i of the (group, KV head, 128-row tile, part of the
// keys) list goes to CTA i * G / n; a CTA issues the copies of its next item
// while the current one computes. S and O live in tensor memory (256 columns).
// Launch 2 (merge): the (row, query head) pairs are split evenly over the CTAs;
// each combines its pairs' part partials in part order.
#include "../../include/eagle.h"
#include "attention_umma.cuh"
#include "kernels.h"

#include <algorithm>

namespace eg {
namespace {

using namespace tc;

constexpr int kUmThreads = 128;
constexpr int kUmMaxGroups = 128;  // groups kept in shared memory
constexpr int kUmMaxCtas = 160;    // partial-slot sizing bound (as the persistent kernel's)

template <int HD>
constexpr size_t um_launch_smem() {
  // staging (1024-byte aligned) + alignment slack + two barriers, TMEM slot, flags + the groups
  return attn::um_smem_bytes<HD>() + 1024 + 64 + kUmMaxGroups * sizeof(Group);
}

template <int HD>
__device__ __forceinline__ void um_launch_layout(uint8_t* raw, uint8_t*& sm, uint64_t*& bars, uint32_t*& tmem_slot,
                                                 volatile int*& abort_flag, Group*& sg) {
  // an offset from the shared array keeps the pointers in the shared address space
  sm = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  bars = reinterpret_cast<uint64_t*>(sm + attn::um_smem_bytes<HD>());
  tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
  abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  sg = reinterpret_cast<Group*>(bars + 4);
}

template <int HD>
__global__ void __launch_bounds__(kUmThreads, 1)
    attn_um_items_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const AttnArgs a, int n_ctas, int slots) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm;
  uint64_t* bars;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  Group* sg;
  um_launch_layout<HD>(smem_raw, sm, bars, tmem_slot, abort_flag, sg);
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = tid; i < a.n_groups; i += kUmThreads) sg[i] = a.groups[i];
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(attn::kUmTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  attn::UmState st;
  st.groups = sg;
  st.sm = sm;
  st.kv_bar = &bars[0];
  st.mma_bar = &bars[1];
  st.tmem = *tmem_slot;
  const attn::UmItems items(a, sg, n_ctas);
  const int n = items.count();
  const int i0 = (int)((long long)blockIdx.x * n / gridDim.x), i1 = (int)((long long)(blockIdx.x + 1) * n / gridDim.x);
  attn::UmItem cur{}, nxt{};
  if (i0 < i1) {
    items.item(i0, cur.chunk, cur.kvh, cur.rt, cur.z);
    if (tid == 0) attn::um_issue<HD>(a, &tmQ, &tmK, &tmV, cur, items.n0, st);
  }
  bool alive = true;
  for (int i = i0; i < i1 && alive; ++i) {
    const bool has_next = i + 1 < i1;
    if (has_next) items.item(i + 1, nxt.chunk, nxt.kvh, nxt.rt, nxt.z);
    alive = attn::attn_item_um<HD>(a, &tmQ, &tmK, &tmV, cur, has_next, nxt, items.n0, slots, st, tid, tid,
                                   abort_flag, EpilogueSync{});
    cur = nxt;
  }
  // no MMA of this CTA is in flight here (every item waited for its own); free tensor memory
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(st.tmem), "r"(attn::kUmTmemCols)
                 : "memory");
  }
}

template <int HD>
__global__ void __launch_bounds__(kUmThreads, 1) attn_um_merge_kernel(const AttnArgs a, int n_ctas, int slots) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm;
  uint64_t* bars;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  Group* sg;
  um_launch_layout<HD>(smem_raw, sm, bars, tmem_slot, abort_flag, sg);
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = tid; i < a.n_groups; i += kUmThreads) sg[i] = a.groups[i];
  __syncthreads();
  const attn::UmItems items(a, sg, n_ctas);  // the items launch's parts request
  const int nm = a.M * a.Hq;
  const int w0 = (int)((long long)blockIdx.x * nm / gridDim.x), w1 = (int)((long long)(blockIdx.x + 1) * nm / gridDim.x);
  // pairs in chunks whose running state and 8 parts' partials fit the staging (large prefill chunks give a
  // CTA hundreds of pairs)
  constexpr int kChunk = (int)(attn::um_smem_bytes<HD>() / ((HD + 2) * 4 + 8 * (HD * 4 + 8)));
  uint32_t par = 0;
  for (int c0 = w0; c0 < w1; c0 += kChunk)
    if (!attn::um_merge_staged<HD>(a, sg, items.n0, c0, min(w1, c0 + kChunk), slots, sm,
                                   (uint32_t)attn::um_smem_bytes<HD>(), &bars[0], &par, tid, abort_flag,
                                   EpilogueSync{}))
      break;
}

template <int HD>
cudaError_t launch_um(const AttnArgs& a, cudaStream_t s) {
  const int G = a.Hq / a.Hkv;
  const long long kv_rows = (long long)a.n_seq * a.Hkv * a.cap;
  const long long q_rows = (long long)a.Hkv * a.M * G;
  if (kv_rows <= 0 || kv_rows > (1ll << 31) - 1 || q_rows > (1ll << 31) - 1) return cudaErrorInvalidValue;
  CUtensorMap tmQ, tmK, tmV;
  if (!make_tmap_f16(&tmQ, a.qg, (int)q_rows, HD, attn::kUmRows) ||
      !make_tmap_f16(&tmK, a.kc, (int)kv_rows, HD, attn::kUmKeys) ||
      !make_tmap_f16(&tmV, a.vc, (int)kv_rows, HD, attn::kUmKeys))
    return cudaErrorInvalidValue;
  const int n_ctas = num_sms();
  if (n_ctas > kUmMaxCtas) return cudaErrorInvalidValue;
  const int slots = attn::um_part_slots(a.max_prefix, a.Hkv, kUmMaxCtas);
  const int smem = (int)um_launch_smem<HD>();
  if (!raise_smem_limit(reinterpret_cast<const void*>(attn_um_items_kernel<HD>), smem) ||
      !raise_smem_limit(reinterpret_cast<const void*>(attn_um_merge_kernel<HD>), smem))
    return cudaErrorInvalidValue;
  // two CTAs per SM (each ~100 KB of shared memory and 256 tensor-memory columns): one item's copies
  // and MMAs overlap the other's softmax and stores
  attn_um_items_kernel<HD><<<2 * n_ctas, kUmThreads, smem, s>>>(tmQ, tmK, tmV, a, n_ctas, slots);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_um_merge_kernel<HD><<<2 * n_ctas, kUmThreads, smem, s>>>(a, n_ctas, slots);
  return cudaGetLastError();
}

// qg[(kvh M + m) G + g][hd] = half(q[m][kvh G + g][:] * scale * log2(e)): the grouped
// half queries the items read (the QKV epilogue writes the same layout).
__global__ void make_qg_kernel(const float* __restrict__ q, int M, int Hq, int Hkv, int hd, float qscale,
                               __half* __restrict__ qg) {
  const int G = Hq / Hkv;
  const long long total = (long long)M * Hq * hd;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int i = (int)(e % hd);
    const long long mh = e / hd;
    const int qh = (int)(mh % Hq), m = (int)(mh / Hq);
    qg[(((long long)(qh / G) * M + m) * G + qh % G) * hd + i] = __float2half_rn(q[e] * qscale);
  }
}

}  // namespace

cudaError_t attention_umma_qg(const float* q, int M, int Hq, int Hkv, int hd, float scale, __half* qg,
                              cudaStream_t s) {
  const long long total = (long long)M * Hq * hd;
  if (total <= 0) return cudaSuccess;
  const long long blocks = std::min<long long>((total + 255) / 256, 152 * 16);
  make_qg_kernel<<<(unsigned)blocks, 256, 0, s>>>(q, M, Hq, Hkv, hd, scale * 1.4426950408889634f, qg);
  return cudaGetLastError();
}

size_t attention_umma_part_bytes(int M, int Hq, int Hkv, int hd, int max_prefix) {
  const size_t slots = (size_t)attn::um_part_slots(max_prefix, Hkv, kUmMaxCtas);
  return (size_t)M * Hq * slots * (hd + 2) * sizeof(float);
}

cudaError_t attention_umma(const AttnArgs& a, cudaStream_t s) {
  if (a.n_groups <= 0 || a.M <= 0) return cudaSuccess;
  if (!a.part || !a.qg || a.Hq % a.Hkv || a.n_groups > kUmMaxGroups) return cudaErrorInvalidValue;
  if (a.hd == 128) return launch_um<128>(a, s);
  if (a.hd == 64) return launch_um<64>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace eg
