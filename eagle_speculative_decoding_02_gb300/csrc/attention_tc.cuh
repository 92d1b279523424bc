// Tree-masked attention on tensor cores (f16 mma.sync m16n8k16, fp32 softmax):
// the work-item and merge bodies, shared by the standalone kernels and the
// persistent layer-stack kernel.
//
// "EAGLE (LLM decoding)", section "How EAGLE works": tree attention verifies
// every draft node in one forward pass. A query row (node j, query head h) of
// group g sees the prefix slots [0, prefix) and the slots prefix + i of the
// tree block whose bit i is set in node j's ancestor mask.
//
// Split-K flash decode: work item (chunk c, KV head and 64-row block, group)
// takes either prefix keys [CKI c, CKI c + CKI) or, for c == ceil(prefix / CKI),
// the tree block, and 64 of the group's rows x G = Hq / Hkv query heads sharing
// that KV head (the GQA rows form the M dimension of the MMA). An item streams
// its keys through shared memory in sub-chunks of CKS keys with cp.async, the
// next sub-chunk in flight while the current one is used (V fragments are read
// transposed with ldmatrix.trans); each of its 4 warps runs one 16-row tile with an online
// softmax and writes an unnormalised partial (max, sum, O). attn_merge_warp
// combines the partials of a row in chunk order. Chunk boundaries are absolute
// slot multiples of CKI, independent of how many rows are verified or batched. The KV cache
// of a bf16 model holds IEEE half values; q (float32, pre-scaled) and the
// probabilities P enter the products rounded to half, so both MMAs are
// f16 x f16 with fp32 accumulation.
#pragma once

#include <cmath>

#include "kernels.h"

namespace eg {
namespace attn {

constexpr int kMaxGroupRows = 128;  // rows of one group (tree rows, or one 128-row prefill block)
constexpr int kPad = 8;             // half padding per shared-memory row (rows 16-byte aligned, conflict-free)
constexpr int kAttnThreads = 128;   // 4 warps, one 16-row tile each
constexpr int kRowBlock = 64;       // GQA rows (node x query head) per work item

// Row blocks per (KV head, group) in the item grid.
__host__ __device__ inline int row_blocks(int Hq, int Hkv) {
  return (kMaxGroupRows * (Hq / Hkv) + kRowBlock - 1) / kRowBlock;
}
// Shared memory of one staging buffer: K and V of CKS keys.
template <int HD, int CKS>
constexpr size_t smem_bytes() { return 2 * (size_t)CKS * (HD + kPad) * sizeof(__half); }

using half = __half;

__device__ __forceinline__ uint32_t ld_b32(const half* p) { return *reinterpret_cast<const uint32_t*>(p); }

__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two floats -> packed half2 (x in the low half).
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

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem), "r"(src_bytes)
               : "memory");
}

// Four 8x8 b16 matrices, transposed, from shared memory (one row address per lane).
__device__ __forceinline__ void ldsm_x4_trans(const half* p, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}

// One work item, run by 128 threads (ranks tid = 0..127, sync() a barrier over
// them): chunk `chunk` (CKI keys) of group `z` for KV head and row block `y`.
// The chunk's keys pass through shared memory CKS at a time: buf holds nbuf
// (1 or 2) staging buffers, each K then V of CKS x (HD + kPad) halves; with two
// the next sub-chunk is staged while the current one is computed. The caller
// syncs before reusing buf. The online-softmax state stays in registers. Each of the 4
// warps owns one 16-row tile of the 64-row block. Returns without work (and
// without syncing) for items past the group's keys or rows.
template <int HD, int CKI, int CKS, typename Sync>
__device__ void attn_item(const AttnArgs& a, int chunk, int y, int z, int n_chunk_slots, half* buf, int nbuf,
                          int tid, Sync sync) {
  static_assert(CKS % 64 == 0 && CKI % CKS == 0 && kRowBlock == 16 * (kAttnThreads / 32), "tiling");
  const Group g = a.groups[z];
  const int rb_count = row_blocks(a.Hq, a.Hkv);
  const int kvh = y / rb_count, rb = y % rb_count;
  const int nck = n_prefix_chunks(g.prefix, CKI);
  const bool block = chunk == nck;
  if (chunk > nck || (block && g.block_len <= 0) || rb * kRowBlock >= g.nrows * (a.Hq / a.Hkv)) return;
  const int key0 = block ? g.prefix : chunk * CKI;
  const int nkeys = block ? min(g.block_len, kMaxGroupRows) : min(CKI, g.prefix - key0);
  const int G = a.Hq / a.Hkv;
  const int R = g.nrows * G;
  const int warp = tid >> 5, lane = tid & 31;
  const int mt = rb * (kRowBlock / 16) + warp;  // this warp's 16-row tile
  const bool active = mt * 16 < R;

  const float sl2 = a.scale * 1.4426950408889634f;  // scores in log2 units
  const int quad = lane >> 2, qi = lane & 3;
  // rows r0 = mt*16 + quad and r1 = r0 + 8 of this tile: (node, head) = (r / G, r % G)
  int node[2], qh[2];
  bool rv[2];
  uint64_t mk0[2], mk1[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = mt * 16 + quad + 8 * i;
    rv[i] = active && r < R;
    node[i] = rv[i] ? r / G : 0;
    qh[i] = kvh * G + (rv[i] ? r % G : 0);
    const int row = g.row0 + node[i];
    mk0[i] = block && rv[i] ? a.mask[2 * row] : 0ull;
    mk1[i] = block && rv[i] ? a.mask[2 * row + 1] : 0ull;
  }
  // q (float32) times the softmax scale in log2 units, rounded to half A fragments
  uint32_t qa[HD / 16][4];
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float* qp = a.q + (((size_t)(g.row0 + node[i])) * a.Hq + qh[i]) * HD;
      // q and the partials are read through L2: in the persistent kernel they were
      // written earlier in the same launch by other SMs
      const float2 x0 = rv[i] ? __ldcg(reinterpret_cast<const float2*>(qp + kk * 16 + qi * 2)) : make_float2(0.f, 0.f);
      const float2 x1 = rv[i] ? __ldcg(reinterpret_cast<const float2*>(qp + kk * 16 + 8 + qi * 2)) : make_float2(0.f, 0.f);
      qa[kk][i] = pack_half2(x0.x * sl2, x0.y * sl2);
      qa[kk][i + 2] = pack_half2(x1.x * sl2, x1.y * sl2);
    }
  }
  float o[HD / 8][4];
#pragma unroll
  for (int dt = 0; dt < HD / 8; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

  const half* Kg = reinterpret_cast<const half*>(a.kc) + (((size_t)g.seq * a.Hkv + kvh) * a.cap + key0) * HD;
  const half* Vg = reinterpret_cast<const half*>(a.vc) + (((size_t)g.seq * a.Hkv + kvh) * a.cap + key0) * HD;
  constexpr int VEC = 8;  // halves per 16-byte vector
  // stage keys kc0 .. kc0 + CKS of the chunk (row-major) into buffer b with
  // asynchronous 16-byte copies, all in flight at once; keys past the chunk are zero-filled
  constexpr int kBuf = CKS * (HD + kPad);  // halves of one K (or V) buffer
  auto stage = [&](int kc0, int b) {
    const int nk = min(CKS, nkeys - kc0);
    half* Kd = buf + b * 2 * kBuf;
    half* Vd = Kd + kBuf;
    for (int e = tid; e < CKS * HD / VEC; e += kAttnThreads) {
      const int key = e / (HD / VEC), d0 = (e % (HD / VEC)) * VEC;
      const int n = key < nk ? 16 : 0;
      const size_t go = (size_t)(kc0 + min(key, nk - 1)) * HD + d0;
      cp_async16(Kd + key * (HD + kPad) + d0, Kg + go, n);
      cp_async16(Vd + key * (HD + kPad) + d0, Vg + go, n);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  const int nsub = (nkeys + CKS - 1) / CKS;
  stage(0, 0);
  for (int j = 0; j < nsub; ++j) {
    const int kc0 = j * CKS;
    const int nk = min(CKS, nkeys - kc0);
    const int bcur = nbuf == 2 ? (j & 1) : 0;
    if (nbuf == 2 && j + 1 < nsub) {
      stage(kc0 + CKS, bcur ^ 1);  // its buffer was freed by the sync that ended sub-chunk j - 1
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    sync();
    const half* Kb = buf + bcur * 2 * kBuf;
    const half* Vb = Kb + kBuf;
    if (active) {
    for (int kb = 0; kb < nk; kb += 64) {
      float s[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const half* kp = Kb + (kb + nt * 8 + quad) * (HD + kPad) + kk * 16 + qi * 2;
          mma16816(s[nt], qa[kk], ld_b32(kp), ld_b32(kp + 8));
        }
      }
      // mask; c-fragment (row quad (+8), chunk key kc0 + kb + nt*8 + qi*2 + {0,1})
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = e >> 1;
          const int key = kc0 + kb + nt * 8 + qi * 2 + (e & 1);
          bool vis = key < nkeys && rv[i];
          if (block && vis) vis = ((key < 64 ? (mk0[i] >> key) : (mk1[i] >> (key - 64))) & 1ull) != 0;
          s[nt][e] = vis ? s[nt][e] : -INFINITY;
          mx[i] = fmaxf(mx[i], s[nt][e]);
        }
      }
      float corr[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
        mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
        const float mn = fmaxf(mrow[i], mx[i]);
        corr[i] = (mn == -INFINITY) ? 1.f : exp2f(mrow[i] - mn);
        mrow[i] = mn;
      }
      float sum[2] = {0.f, 0.f};
      uint32_t pa[4][4];  // P as half A fragments
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = e >> 1;
          const float p = (s[nt][e] == -INFINITY) ? 0.f : exp2f(s[nt][e] - mrow[i]);
          s[nt][e] = p;
          sum[i] += p;
        }
        // P as the A operand of P.V: keys 16*kk2 .. of this 64-key block
        const int kk2 = nt >> 1, hi = nt & 1;
        pa[kk2][0 + 2 * hi] = pack_half2(s[nt][0], s[nt][1]);
        pa[kk2][1 + 2 * hi] = pack_half2(s[nt][2], s[nt][3]);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        sum[i] += __shfl_xor_sync(0xffffffffu, sum[i], 1);
        sum[i] += __shfl_xor_sync(0xffffffffu, sum[i], 2);
        lrow[i] = lrow[i] * corr[i] + sum[i];
      }
#pragma unroll
      for (int dt = 0; dt < HD / 8; ++dt) {
        o[dt][0] *= corr[0];
        o[dt][1] *= corr[0];
        o[dt][2] *= corr[1];
        o[dt][3] *= corr[1];
      }
      // B fragments of V (k = key, n = dim) from the row-major V tile with ldmatrix.trans:
      // lane l addresses row (key) kb + 16 kk2 + 8 ((l >> 3) & 1) + (l & 7) of dim tile dt + (l >> 4)
#pragma unroll
      for (int kk2 = 0; kk2 < 4; ++kk2) {
#pragma unroll
        for (int dt = 0; dt < HD / 8; dt += 2) {
          const int key = kb + kk2 * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
          const half* vp = Vb + key * (HD + kPad) + (dt + (lane >> 4)) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_trans(vp, b0, b1, b2, b3);
          mma16816(o[dt], pa[kk2], b0, b1);
          mma16816(o[dt + 1], pa[kk2], b2, b3);
        }
      }
    }
    }  // active
    sync();  // every warp is done with buffer bcur before it is staged again
    if (nbuf == 1 && j + 1 < nsub) stage(kc0 + CKS, 0);
  }
  if (!active) return;
  const PartLayout pl{a.part, a.M * a.Hq, n_chunk_slots, HD};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (!rv[i]) continue;
    const int w = (g.row0 + node[i]) * a.Hq + qh[i];
    if (qi == 0) *reinterpret_cast<float2*>(pl.ml(chunk, w)) = make_float2(mrow[i], lrow[i]);
#pragma unroll
    for (int dt = 0; dt < HD / 8; ++dt)
      *reinterpret_cast<float2*>(pl.o(chunk, w, dt / 4) + (dt % 4) * 8 + qi * 2) =
          make_float2(o[dt][2 * i], o[dt][2 * i + 1]);
  }
}

// One warp per (row, query head) w < M * Hq: combine the row's chunk partials
// (max m_c, sum l_c, unnormalised O_c) in chunk order. Chunks are taken 16 at a
// time with every load of the block in flight at once, the first block's loads
// issued before the row's group (and so its chunk count) is known: slots past
// the group's chunks hold stale but finite values and are masked out. With M
// the running maximum, weights exp2(m_c - M) scale l_c and O_c, and the running
// sums are rescaled when a later block raises M.
template <int HD, int CKI>
__device__ void attn_merge_warp(const AttnArgs& a, int w, int lane, int n_chunk_slots) {
  constexpr int kB = 16;
  const PartLayout pl{a.part, a.M * a.Hq, n_chunk_slots, HD};
  float mc[kB], lc[kB], oc[kB][HD / 32];
  auto load = [&](int c0) {
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const bool in = c0 + j < n_chunk_slots;
      const float2 ml = in ? __ldcg(reinterpret_cast<const float2*>(pl.ml(c0 + j, w))) : make_float2(-INFINITY, 0.f);
      mc[j] = ml.x;
      lc[j] = ml.y;
#pragma unroll
      for (int i = 0; i < HD / 32; ++i) oc[j][i] = in ? __ldcg(pl.o(c0 + j, w, i) + lane) : 0.f;
    }
  };
  load(0);
  const int row = w / a.Hq, qh = w % a.Hq;
  const Group g = a.groups[a.row_grp ? a.row_grp[row] : 0];
  const int nck = n_prefix_chunks(g.prefix, CKI) + (g.block_len > 0 ? 1 : 0);
  float M = -INFINITY, L = 0.f;
  float acc[HD / 32];
#pragma unroll
  for (int i = 0; i < HD / 32; ++i) acc[i] = 0.f;
  for (int c0 = 0; c0 < nck; c0 += kB) {
    if (c0 > 0) load(c0);
#pragma unroll
    for (int j = 0; j < kB; ++j)
      if (c0 + j >= nck) mc[j] = -INFINITY;  // past the group's chunks
    float Mb = M;
#pragma unroll
    for (int j = 0; j < kB; ++j) Mb = fmaxf(Mb, mc[j]);
    if (Mb == -INFINITY) continue;  // nothing visible yet
    const float r = M == -INFINITY ? 0.f : exp2f(M - Mb);
    L *= r;
#pragma unroll
    for (int i = 0; i < HD / 32; ++i) acc[i] *= r;
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const bool use = mc[j] != -INFINITY;
      const float wgt = use ? exp2f(mc[j] - Mb) : 0.f;
      L += use ? wgt * lc[j] : 0.f;
#pragma unroll
      for (int i = 0; i < HD / 32; ++i) acc[i] += use ? wgt * oc[j][i] : 0.f;
    }
    M = Mb;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const size_t ob = ((size_t)row * a.Hq + qh) * HD;
#pragma unroll
  for (int i = 0; i < HD / 32; ++i) store_hilo<bf16>(reinterpret_cast<bf16*>(a.o), a.o_lo, ob + lane + 32 * i, acc[i] * inv);
}

}  // namespace attn
}  // namespace eg
