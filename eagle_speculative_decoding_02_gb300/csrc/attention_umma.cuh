// Tree-masked attention work item on the 5th-generation tensor cores
// (tcgen05.mma, operands in shared memory, scores and output in tensor memory),
// run by the four epilogue warps of the persistent layer-stack kernel.
//
// "EAGLE (LLM decoding)", section "How EAGLE works": tree attention verifies
// every draft node in one forward pass; a query row (node j, query head h) sees
// the prefix slots [0, prefix) and the slots prefix + i of the tree block whose
// bit i is set in node j's ancestor mask.
//
// Split-K flash decode, one item = (chunk of 128 keys, KV head, tile of 128 GQA
// rows, group). The GQA rows (node x query head sharing the KV head) are the
// MMA's M dimension, one tensor-memory lane per row, so each thread owns one row:
//
//   1. TMA brings the tile's query rows (q * softmax_scale * log2(e) as half,
//      written grouped by KV head by the QKV epilogue) and the chunk's K and V
//      rows (fp16 KV cache) into shared memory, 128-byte swizzled.
//   2. S = Q K^T: HD / 16 MMAs (M = 128, N = 128 keys), fp32 in TMEM columns
//      [0, 128).
//   3. Each thread reads its S row twice from TMEM (max, then exp2 and sum),
//      masks it, and writes P = exp2(S - max) rounded to half into a K-major P
//      tile that reuses the K buffer (the K rows are dead once S is complete;
//      the buffer holds 128 x max(HD, 128) halves).
//   4. O = P V: 8 MMAs (N = HD), V read in place as an MN-major operand (its rows
//      are keys, contiguous in head dimension); fp32 in TMEM columns [128, 256).
//   5. The row's unnormalised partial (O, max, sum) goes out for
//      attn_merge_warp, in the layout the mma.sync path writes too. The next
//      item's copies are issued as soon as the MMAs are done, so they overlap
//      this step.
//
// Precision matches the mma.sync path: half q, K, P and V, fp32 accumulation.
#pragma once

#include "attention_tc.cuh"
#include "tc_ptx.cuh"

namespace eg {
namespace attn {

using namespace tc;

constexpr int kUmRows = 128;  // GQA rows of an item (one TMEM lane each)
constexpr int kUmKeys = 128;  // keys of an item
constexpr uint32_t kUmAtom = kUmRows * 128;  // bytes of one 64-column swizzle atom of a 128-row half tile
constexpr uint32_t kUmColS = 0;              // TMEM column of S
constexpr uint32_t kUmColO = 128;            // TMEM column of O
constexpr uint32_t kUmTmemCols = 256;        // tensor-memory columns an item needs

// Row tiles of a group of nrows tree rows with G query heads per KV head.
__host__ __device__ inline int um_row_tiles(int nrows, int G) { return (nrows * G + kUmRows - 1) / kUmRows; }
// Shared memory of an item: Q and V tiles (128 rows x HD halves), then the K
// tile that P (128 rows x 128 keys) later overwrites.
template <int HD>
constexpr size_t um_kp_bytes() { return (size_t)kUmRows * (HD > kUmKeys ? HD : kUmKeys) * 2; }
template <int HD>
constexpr size_t um_smem_bytes() { return 2 * (size_t)kUmRows * HD * 2 + um_kp_bytes<HD>(); }

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled atom
// (the layout TMA's 128B swizzle writes and the K-major descriptor reads).
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// MN-major operand of 128-byte-swizzled atoms: 8-row (K) groups sbo bytes apart,
// 64-element (MN) atoms lbo bytes apart.
__device__ __forceinline__ uint64_t sw128_desc_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16 with half A and B, fp32 D, M = 128, N = n;
// b_mn: B is MN-major.
__host__ __device__ constexpr uint32_t idesc_f16(int n, bool b_mn) {
  return (1u << 4) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// 2^x by the PTX approximation (relative error about 2^-22; the probabilities are
// rounded to half right after). 2^-inf = +0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Per-CTA state of the items: staging region, barriers and their phase parities.
struct UmState {
  uint8_t* sm;         // um_smem_bytes<HD>() bytes, 1024-byte aligned
  uint64_t* kv_bar;    // TMA of K and V
  uint64_t* mma_bar;   // tcgen05.commit of S, then of O
  uint32_t tmem;       // tensor-memory base (lane 0, column 0)
  uint32_t kv_par = 0, mma_par = 0;
};

// An item: chunk of the group's keys (the last one is the tree block), KV head,
// 128-row tile, group.
struct UmItem {
  int chunk, kvh, rt, z;
};

// Thread 0 of the item's 128: issue the TMA copies of item `it`'s Q, K and V
// tiles onto st.kv_bar (the buffers must be free: no MMA still reading them, and
// every thread's generic writes to them fenced and past a barrier). tmQ, tmK,
// tmV: 2D maps (box 128 rows x 64 halves, 128-byte swizzle) of a.qg as
// [Hkv * M * G][HD] and of the K / V caches as [n_seq * Hkv * cap][HD].
template <int HD>
__device__ void um_issue(const AttnArgs& a, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                         const CUtensorMap* tmV, const UmItem& it, const UmState& st) {
  const Group g = a.groups[it.z];
  const int G = a.Hq / a.Hkv;
  const int nck = n_prefix_chunks(g.prefix, kUmKeys);
  const int key0 = it.chunk == nck ? g.prefix : it.chunk * kUmKeys;
  uint8_t* sQ = st.sm;
  uint8_t* sV = sQ + (size_t)kUmRows * HD * 2;
  uint8_t* sK = sV + (size_t)kUmKeys * HD * 2;
  // q and this layer's new K / V rows were written by other SMs' generic stores
  // earlier in the launch; the copies read them through the async proxy
  asm volatile("fence.proxy.async.global;" ::: "memory");
  mbar_expect_tx(st.kv_bar, (uint32_t)(3 * kUmRows * HD * 2));
  const int ykv = (g.seq * a.Hkv + it.kvh) * a.cap + key0;
  const int yq = (it.kvh * a.M + g.row0) * G + it.rt * kUmRows;
#pragma unroll
  for (int h = 0; h < HD / 64; ++h) {
    tma_load_2d(sQ + h * kUmAtom, tmQ, st.kv_bar, h * 64, yq);
    tma_load_2d(sK + h * kUmAtom, tmK, st.kv_bar, h * 64, ykv);
    tma_load_2d(sV + h * kUmAtom, tmV, st.kv_bar, h * 64, ykv);
  }
}

// One item, run by 128 threads: tid 0..127 (tid 0 issues the copies and MMAs),
// row = the TMEM lane this thread may read (its warp's lane quarter x 32 + lane)
// and thus its row of the tile. sync() is a barrier over the 128 threads. The
// item's copies were issued (um_issue); once its MMAs are done and before its
// partials go out, thread 0 issues those of `next` when has_next. The caller
// passes only items with keys and rows. Returns false on a timeout (status set,
// abort raised).
template <int HD, typename Sync>
__device__ bool attn_item_um(const AttnArgs& a, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                             const CUtensorMap* tmV, const UmItem& cur, bool has_next, const UmItem& next,
                             int n_chunk_slots, UmState& st, int tid, int row, volatile int* abort_flag,
                             Sync sync) {
  static_assert(HD == 64 || HD == 128, "head dim");
  const Group g = a.groups[cur.z];
  const int G = a.Hq / a.Hkv;
  const int R = g.nrows * G;
  const int nck = n_prefix_chunks(g.prefix, kUmKeys);
  const bool block = cur.chunk == nck;
  const int key0 = block ? g.prefix : cur.chunk * kUmKeys;
  const int nkeys = block ? min(g.block_len, kUmKeys) : min(kUmKeys, g.prefix - key0);
  const int r = cur.rt * kUmRows + row;
  const bool rv = r < R;
  const int node = rv ? r / G : 0;
  const int qh = cur.kvh * G + (rv ? r % G : 0);
  uint8_t* sQ = st.sm;
  uint8_t* sV = sQ + (size_t)kUmRows * HD * 2;
  uint8_t* sK = sV + (size_t)kUmKeys * HD * 2;  // K, then P
  const uint32_t lane_base = (uint32_t)(row & ~31) << 16;

  // visibility of this row's keys, 32 per word: key < nkeys, and in the tree
  // block the node's ancestor bit
  uint32_t vis[kUmKeys / 32];
  {
    uint64_t mk0 = ~0ull, mk1 = ~0ull;
    if (block && rv) {
      mk0 = a.mask[2 * (g.row0 + node)];
      mk1 = a.mask[2 * (g.row0 + node) + 1];
    }
#pragma unroll
    for (int b = 0; b < kUmKeys / 32; ++b) {
      uint32_t w = (uint32_t)((b < 2 ? mk0 : mk1) >> ((b & 1) * 32));
      const int left = nkeys - 32 * b;
      w &= left >= 32 ? ~0u : (left <= 0 ? 0u : (1u << left) - 1u);
      vis[b] = rv ? w : 0u;
    }
  }

  // 1. S = Q K^T once the copies have landed
  bool ok = true;
  if (tid == 0) {
    ok = mbar_wait(st.kv_bar, st.kv_par, abort_flag, a.status);
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kUmAtom + (kk & 3) * 32;
        umma(st.tmem + kUmColS, sw128_desc(smem_u32(sQ) + off), sw128_desc(smem_u32(sK) + off),
             idesc_f16(kUmKeys, false), kk > 0 ? 1u : 0u);
      }
      umma_commit(st.mma_bar);
    }
  }
  st.kv_par ^= 1;
  ok = epi_all(tid != 0 || ok);
  if (ok) ok = epi_all(mbar_wait(st.mma_bar, st.mma_par, abort_flag, a.status));
  st.mma_par ^= 1;
  if (!ok) return false;  // (a timed-out wait leaves the CTA to abort; no MMA is left issued)
  tc_fence_after();

  // 2. masked softmax of this row (scores are in log2 units); P (half) into the K buffer
  float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
  for (int b = 0; b < kUmKeys / 32; b += 2) {
    float s[2][32];
    tmem_ld64(st.tmem + lane_base + kUmColS + 32 * b, s[0], s[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t w = vis[b + h];
      if (w == ~0u) {  // every key of the word visible (prefix chunks)
#pragma unroll
        for (int i = 0; i < 32; ++i) m4[i & 3] = fmaxf(m4[i & 3], s[h][i]);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) m4[i & 3] = fmaxf(m4[i & 3], ((w >> i) & 1u) ? s[h][i] : -INFINITY);
      }
    }
  }
  const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
  const float mxs = mx == -INFINITY ? 0.f : mx;  // a row with no visible key: every p is 0
  float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int b = 0; b < kUmKeys / 32; b += 2) {
    float s[2][32];
    tmem_ld64(st.tmem + lane_base + kUmColS + 32 * b, s[0], s[1]);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t w = vis[b + h];
      if (w == ~0u) {
#pragma unroll
        for (int i = 0; i < 32; ++i) s[h][i] = ex2_approx(s[h][i] - mxs);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) s[h][i] = ((w >> i) & 1u) ? ex2_approx(s[h][i] - mxs) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) l4[i & 3] += s[h][i];
      const int bb = b + h;
#pragma unroll
      for (int c = 0; c < 4; ++c) {  // keys 32 bb + 8 c .. + 7: chunk (4 bb + c) % 8 of atom bb / 2
        uint4 hv;
        hv.x = pack_half2(s[h][8 * c + 0], s[h][8 * c + 1]);
        hv.y = pack_half2(s[h][8 * c + 2], s[h][8 * c + 3]);
        hv.z = pack_half2(s[h][8 * c + 4], s[h][8 * c + 5]);
        hv.w = pack_half2(s[h][8 * c + 6], s[h][8 * c + 7]);
        *reinterpret_cast<uint4*>(sK + (bb >> 1) * kUmAtom + sw128_off(row, ((bb & 1) << 2) + c)) = hv;
      }
    }
  }
  const float sum = (l4[0] + l4[1]) + (l4[2] + l4[3]);
  fence_proxy_async_smem();  // P is read by the tensor cores
  tc_fence_before();
  sync();

  // 3. O = P V
  if (tid == 0) {
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < kUmKeys / 16; ++kk) {
      const uint32_t offp = (kk >> 2) * kUmAtom + (kk & 3) * 32;
      umma(st.tmem + kUmColO, sw128_desc(smem_u32(sK) + offp),
           sw128_desc_mn(smem_u32(sV) + kk * 2048, kUmAtom, 1024), idesc_f16(HD, true), kk > 0 ? 1u : 0u);
    }
    umma_commit(st.mma_bar);
  }
  ok = epi_all(mbar_wait(st.mma_bar, st.mma_par, abort_flag, a.status));
  st.mma_par ^= 1;
  if (!ok) return false;
  tc_fence_after();
  // every tile is free again: the next item's copies overlap this item's output
  if (tid == 0 && has_next) um_issue<HD>(a, tmQ, tmK, tmV, next, st);

  // 4. the row's partial (tcgen05.ld is warp-wide: every lane loads)
  const PartLayout pl{a.part, a.M * a.Hq, n_chunk_slots, HD};
  const int w = (g.row0 + node) * a.Hq + qh;
#pragma unroll 1
  for (int b = 0; b < HD / 32; b += 2) {
    float o[2][32];
    tmem_ld64(st.tmem + lane_base + kUmColO + 32 * b, o[0], o[1]);
    if (rv) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float4* dst = reinterpret_cast<float4*>(pl.o(cur.chunk, w, b + h));
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_float4(o[h][4 * i], o[h][4 * i + 1], o[h][4 * i + 2], o[h][4 * i + 3]);
      }
    }
  }
  if (rv) *reinterpret_cast<float2*>(pl.ml(cur.chunk, w)) = make_float2(mx, sum);
  tc_fence_before();
  return true;
}

}  // namespace attn
}  // namespace eg
