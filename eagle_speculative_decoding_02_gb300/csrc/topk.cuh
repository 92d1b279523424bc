// Merge of the LM-head epilogue's per-tile records into each row's top-k and
// log-sum-exp ("EAGLE (LLM decoding)", section "How EAGLE works": the draft head
// reuses the target's LM head and expands the top-k tokens of each node; verify
// takes the target's top-1 per tree row). The GEMM epilogue leaves, per (vocab
// tile, row), the tile's k best logits (value descending, index ascending) and
// the tile's (max, sum of exp(x - max)); this merge combines them over the tiles.
// Used by the standalone merge kernel and by the persistent layer-stack kernel
// (after its LM-head phase, one CTA per row).
#pragma once

#include "common.cuh"

namespace eg {

// Records of one LM-head GEMM over M rows and ntiles vocab tiles: entry (t, m)
// at t * M + m (val / idx: k entries each), and where the merged rows go.
struct TopkMerge {
  const float* val = nullptr;
  const int* idx = nullptr;
  const float* mx = nullptr;
  const float* sum = nullptr;
  int ntiles = 0, M = 0, k = 0;  // k == 0: no merge
  int* out_idx = nullptr;        // [M][k]: -1 where fewer than k candidates exist
  float* out_val = nullptr;      // [M][k] or NULL
  float* out_lse = nullptr;      // [M] or NULL
};

// Row m by NT threads (tid 0..NT-1, NT a multiple of 32): out_idx / out_val get
// the row's k best (value descending, index ascending) and out_lse its
// log-sum-exp. red: 4 * NT / 32 words of shared memory; sync(): a barrier over
// the NT threads. The records are read through L2 (ld.global.cg): inside one
// launch other SMs wrote them, and L1 is not coherent with their stores.
template <int NT, typename Sync>
__device__ void topk_merge_row(const TopkMerge& g, int m, int tid, float* red, Sync sync) {
  constexpr int NW = NT / 32;
  float* red_m = red;
  float* red_s = red + NW;
  float* sv = red + 2 * NW;
  int* si = reinterpret_cast<int*>(red + 3 * NW);
  const int ntiles = g.ntiles, M = g.M, k = g.k;
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
  // each thread keeps the k best of its candidates (value desc, index asc), sorted, in registers
  float lv[kMaxTopK];
  int li[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    lv[j] = -INFINITY;
    li[j] = 0x7fffffff;
  }
  constexpr int kU = 2;
  for (int t0 = tid; t0 < ntiles; t0 += kU * NT) {
    float tm[kU], ts[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int t = t0 + u * NT;
      const size_t r = (size_t)t * M + m;
      tm[u] = t < ntiles ? __ldcg(g.mx + r) : -INFINITY;
      ts[u] = t < ntiles ? __ldcg(g.sum + r) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) combine(rm, rs, tm[u], ts[u]);
    for (int u = 0; u < kU; ++u) {
      const int t = t0 + u * NT;
      if (t >= ntiles) break;
      // the tile's best is its max: nothing of the tile enters unless that does
      if (!(tm[u] >= lv[k - 1])) continue;
      const size_t base = ((size_t)t * M + m) * k;
      float cv[kMaxTopK];
      int cx[kMaxTopK];
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j) {  // the tile's candidates, all loads in flight
        cv[j] = j < k ? __ldcg(g.val + base + j) : -INFINITY;
        cx[j] = j < k ? __ldcg(g.idx + base + j) : -1;
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
  // (max, sum) over the threads: warps by shuffles, then the warps in order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, rm, o), os = __shfl_xor_sync(0xffffffffu, rs, o);
    combine(rm, rs, om, os);
  }
  if ((tid & 31) == 0) {
    red_m[tid >> 5] = rm;
    red_s[tid >> 5] = rs;
  }
  sync();
  if (tid == 0 && g.out_lse) {
    float gm = red_m[0], gs = red_s[0];
    for (int w = 1; w < NW; ++w) combine(gm, gs, red_m[w], red_s[w]);
    g.out_lse[m] = gm + __logf(gs);
  }

  // k rounds of an arg-max over the heads of the sorted lists
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
    sync();
    if ((tid & 31) == 0) {
      sv[tid >> 5] = bv;
      si[tid >> 5] = bi;
    }
    sync();
    bv = sv[0];
    bi = si[0];
    for (int w = 1; w < NW; ++w)
      if (sv[w] > bv || (sv[w] == bv && si[w] < bi)) {
        bv = sv[w];
        bi = si[w];
      }
    if (mine == bi && head < k) ++head;  // indices are unique: exactly one list owns the winner
    if (tid == 0) {
      g.out_idx[(size_t)m * k + r] = bi == 0x7fffffff ? -1 : bi;
      if (g.out_val) g.out_val[(size_t)m * k + r] = bv;
    }
  }
  sync();  // red is free again
}

}  // namespace eg
