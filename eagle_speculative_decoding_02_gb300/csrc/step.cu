// Per-step kernels of the speculative loop: row metadata for each forward
// phase, static and EAGLE-2 draft trees, greedy acceptance and in-place KV
// compaction. All are latency kernels (one block per sequence or per row).
#include "step.h"

namespace eg {
namespace {

__device__ __forceinline__ void causal_mask(int i, uint64_t* m) {
  // bits 0..i set
  if (i < 64) {
    m[0] = (i == 63) ? ~0ull : ((1ull << (i + 1)) - 1ull);
    m[1] = 0ull;
  } else {
    m[0] = ~0ull;
    m[1] = (i == 127) ? ~0ull : ((1ull << (i - 63)) - 1ull);
  }
}

// Prefill chunk [c0, c0 + CL) of every prompt. Target rows read prompt token
// c0+i at slot c0+i; draft rows take token c0+i+1 (the shifted sequence) and
// skip the last prompt position, whose next token is not known yet.
__global__ void setup_prefill_kernel(const int* __restrict__ prompt, int P, int c0, int CL, int B, int draft,
                                     Rows rows, Group* groups) {
  pdl_wait();
  pdl_trigger();
  const int G = (CL + 127) / 128;
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m < B * CL) {
    const int b = m / CL, i = m % CL, p = c0 + i;
    int tok = prompt[(size_t)b * P + p], slot = p;
    if (draft) {
      if (p + 1 < P) {
        tok = prompt[(size_t)b * P + p + 1];
      } else {
        tok = 0;
        slot = -1;
      }
    }
    rows.seq[m] = b;
    rows.pos[m] = p;
    rows.slot[m] = slot;
    rows.tok[m] = tok;
    rows.fsrc[m] = m;
    rows.grp[m] = b * G + i / 128;
    causal_mask(i % 128, rows.mask + 2 * m);
  }
  if (m < B * G) {
    const int b = m / G, sub = m % G;
    Group g;
    g.seq = b;
    g.row0 = b * CL + sub * 128;
    g.nrows = min(128, CL - sub * 128);
    g.prefix = c0 + sub * 128;
    g.block_len = g.nrows;
    groups[m] = g;
  }
}

// Catch-up rows of the draft head: per sequence D1 rows, the first c valid.
__global__ void setup_catchup_kernel(State st, Rows rows, Group* groups) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, i = threadIdx.x;
  const int L = st.L[b], c = st.c[b];
  if (i < st.D1) {
    const int m = b * st.D1 + i;
    const bool valid = i < c;
    rows.seq[m] = b;
    rows.pos[m] = valid ? L - c + i : 0;
    rows.slot[m] = valid ? L - c + i : -1;
    rows.tok[m] = valid ? st.pend_tok[b * st.D1 + i] : 0;
    rows.fsrc[m] = m;
    rows.grp[m] = b;
    if (valid) {
      causal_mask(i, rows.mask + 2 * m);
    } else {
      rows.mask[2 * m] = 0ull;
      rows.mask[2 * m + 1] = 0ull;
    }
  }
  if (i == 0) {
    Group g;
    g.seq = b;
    g.row0 = b * st.D1;
    g.nrows = st.D1;
    g.prefix = L - c;
    g.block_len = c;
    groups[b] = g;
  }
}

// Is row j of a sequence's tree (rows at `base`) consistent: root at row 0,
// parents earlier in BFS order, depth = parent's depth + 1, ancestor mask =
// parent's mask + its own bit, and a token distinct from its earlier siblings'
// (padding rows carry token -1 and are exempt)?
__device__ bool tree_row_ok(const TreeOut& tree, int base, int j) {
  const int m = base + j;
  const uint64_t a0 = tree.anc[2 * m], a1 = tree.anc[2 * m + 1];
  if (j == 0) return tree.parent[m] == -1 && tree.depth[m] == 0 && a0 == 1ull && a1 == 0ull;
  const int p = tree.parent[m];
  if (p < 0 || p >= j) return false;
  const int dj = tree.depth[m];
  if (dj != tree.depth[base + p] + 1) return false;
  uint64_t e0 = tree.anc[2 * (base + p)], e1 = tree.anc[2 * (base + p) + 1];
  if (j < 64) e0 |= 1ull << j; else e1 |= 1ull << (j - 64);
  if (a0 != e0 || a1 != e1) return false;
  const int tok = tree.tokens[m];
  if (tok >= 0)
    for (int i = 1; i < j; ++i)
      if (tree.parent[base + i] == p && tree.tokens[base + i] == tok) return false;
  return true;
}

// Verify rows: tree row j of sequence b at position L + depth(j), KV slot L + j.
__global__ void setup_verify_kernel(State st, TreeOut tree, Rows rows, Group* groups, Group* groups_local, int spc) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const int NR = tree.n_rows;
  const int L = st.L[b];
  const bool fits = L + NR <= st.cap;
  if (!fits && threadIdx.x == 0) set_status(st.status, kStCapacity);
  for (int j = threadIdx.x; j < NR; j += blockDim.x)
    if (!tree_row_ok(tree, b * NR, j)) set_status(st.status, kStInvalid);
  for (int j = threadIdx.x; j < NR; j += blockDim.x) {
    const int m = b * NR + j;
    rows.seq[m] = b;
    const int tok = tree.tokens[m];
    rows.pos[m] = fits ? L + tree.depth[m] : 0;
    rows.slot[m] = fits && tok >= 0 ? L + j : -1;  // padding rows write no K / V
    rows.tok[m] = (tok >= 0 && tok < st.V) ? tok : 0;  // padding nodes carry -1
    rows.fsrc[m] = m;
    rows.grp[m] = b;
    rows.mask[2 * m] = tree.anc[2 * m];
    rows.mask[2 * m + 1] = tree.anc[2 * m + 1];
  }
  // the attention group holds the tree's real rows: a drafted tree of fewer
  // nodes than rows ends in padding rows (token -1), which no row attends to
  // and accept never takes
  __shared__ int s_real;
  if (threadIdx.x == 0) s_real = NR;
  __syncthreads();
  for (int j = 1 + threadIdx.x; j < NR; j += blockDim.x)
    if (tree.tokens[b * NR + j] < 0) atomicMin(&s_real, j);
  __syncthreads();
  for (int j = s_real + threadIdx.x; j < NR; j += blockDim.x)  // padding rows come last
    if (tree.tokens[b * NR + j] >= 0) set_status(st.status, kStInvalid);
  if (threadIdx.x == 0) {
    Group g;
    g.seq = b;
    g.row0 = b * NR;
    g.nrows = s_real;
    g.prefix = fits ? L : 0;
    g.block_len = fits ? s_real : 0;
    groups[b] = g;
    g.row0 = (spc > 0 ? b % spc : b) * NR;
    groups_local[b] = g;
  }
}

// After the last prefill chunk: first new token per sequence and the initial state.
__global__ void prefill_finish_kernel(State st, const int* __restrict__ root_idx, const float* __restrict__ h_tgt,
                                      const float* __restrict__ h_low, const float* __restrict__ h_mid, int CL, int P,
                                      int* root_out) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const int root = root_idx[b];
  const size_t src = ((size_t)b * CL + CL - 1) * st.d, dst = (size_t)b * st.D1 * st.d;
  for (int n = threadIdx.x; n < st.d; n += blockDim.x) {
    st.pend_feat[dst + n] = h_tgt[src + n];
    if (st.pend_low) {
      st.pend_low[dst + n] = h_low[src + n];
      st.pend_mid[dst + n] = h_mid[src + n];
    }
  }
  if (threadIdx.x == 0) {
    st.L[b] = P;
    st.c[b] = 1;
    st.root[b] = root;
    st.pend_tok[b * st.D1] = root;
    st.n_out[b] = 1;
    st.out[(size_t)b * st.out_cap] = root;
    st.acc_len[b] = 0;
    st.L_prev[b] = P;
    if (root_out) root_out[b] = root;
  }
}

__global__ void set_root_tree_kernel(State st, TreeOut tree) {
  pdl_wait();
  pdl_trigger();
  const int b = threadIdx.x;
  if (b < st.B) {
    const int m = b * tree.n_rows;
    tree.tokens[m] = st.root[b];
    tree.parent[m] = -1;
    tree.depth[m] = 0;
    tree.anc[2 * m] = 1ull;
    tree.anc[2 * m + 1] = 0ull;
  }
}

// ---------------------------------------------------------------- static tree
__global__ void static_level_kernel(State st, StaticTopo topo, int t, const int* __restrict__ topk_idx,
                                    const float* __restrict__ topk_val, const float* __restrict__ lse,
                                    Level catchup, Level prev, Level next, TreeOut tree, Rows rows,
                                    Group* groups, int S) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const int NR = topo.n_rows;
  const int L = st.L[b], c = st.c[b];
  const int root_row = catchup.base + b * catchup.per_seq + c - 1;
  // tokens of depth-t nodes, and their cumulative draft log-confidence (the
  // parent's, written by the previous level, plus the node's own log-probability)
  for (int j = threadIdx.x; j < NR; j += blockDim.x) {
    if (j == 0 && t == 1) {
      tree.tokens[b * NR] = st.root[b];
      if (tree.score) tree.score[b * NR] = 0.f;
    }
    if (topo.depth[j] != t) continue;
    const int p = topo.parent[j];
    const int prow = (p == 0) ? root_row : prev.base + b * prev.per_seq + topo.lrow[p];
    const size_t at = (size_t)prow * topo.k + topo.rank[j];
    tree.tokens[b * NR + j] = topk_idx[at];
    if (tree.score) tree.score[b * NR + j] = (p == 0 ? 0.f : tree.score[b * NR + p]) + (topk_val[at] - lse[prow]);
  }
  if (next.per_seq == 0) return;
  __syncthreads();
  // rows of the depth-t draft forward: its non-leaf nodes
  const int n = topo.level_count[t];
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int j = topo.level_nodes[t * NR + i];
    const int p = topo.parent[j];
    const int m = b * n + i;
    rows.seq[m] = b;
    rows.pos[m] = L + t - 1;
    rows.slot[m] = L + topo.sidx[j];
    rows.tok[m] = tree.tokens[b * NR + j];
    rows.fsrc[m] = (p == 0) ? root_row : prev.base + b * prev.per_seq + topo.lrow[p];
    rows.grp[m] = b;
    rows.mask[2 * m] = topo.smask[j];
    rows.mask[2 * m + 1] = 0ull;
  }
  if (threadIdx.x == 0) {
    Group g;
    g.seq = b;
    g.row0 = b * n;
    g.nrows = n;
    g.prefix = L;
    g.block_len = S;
    groups[b] = g;
  }
}

// ---------------------------------------------------------------- EAGLE-2
__device__ __forceinline__ unsigned int desc_key(float score) {
  // Ascending unsigned order of this key = descending score (+0 and -0 equal).
  const float x = -score + 0.0f;
  const unsigned int u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned long long sort_key(float score, int cid) {
  return ((unsigned long long)desc_key(score) << 32) | (unsigned int)cid;
}

// Block-wide bitonic sort of n (power of two, <= 1024) 64-bit keys with payloads.
__device__ void bitonic_sort(unsigned long long* key, int* val, int n) {
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;
          if ((key[i] > key[j]) == up) {
            const unsigned long long tk = key[i];
            key[i] = key[j];
            key[j] = tk;
            const int tv = val[i];
            val[i] = val[j];
            val[j] = tv;
          }
        }
      }
    }
  }
  __syncthreads();
}

constexpr int kPoolSort = 1024;

__global__ void __launch_bounds__(256) eagle2_level_kernel(State st, Pool pool, int t, int depth, int k,
                                                           float ln_tau, const int* __restrict__ topk_idx,
                                                           const float* __restrict__ topk_val,
                                                           const float* __restrict__ lse, Level catchup,
                                                           Level prev, Level next, Rows rows, Group* groups,
                                                           int S) {
  pdl_wait();
  pdl_trigger();
  __shared__ unsigned long long key[128];
  __shared__ int val[128];
  __shared__ int s_first, s_n;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int L = st.L[b], c = st.c[b];
  const size_t pb = (size_t)b * pool.cap;
  if (t == 1) {
    // children of the root: the catch-up row's top-k
    const int r = catchup.base + b * catchup.per_seq + c - 1;
    if (tid < k) {
      const int e = tid;
      pool.score[pb + e] = topk_val[(size_t)r * k + tid] - lse[r];
      pool.token[pb + e] = topk_idx[(size_t)r * k + tid];
      pool.parent[pb + e] = -1;
      pool.depth[pb + e] = 1;
      pool.cid[pb + e] = (1 << 16) | tid;
      pool.frow[pb + e] = -1;
      pool.smask[pb + e] = 0ull;
    }
    if (tid == 0) {
      pool.count[b] = k;
      s_first = 0;
      s_n = k;
    }
  } else {
    const int nf = pool.nfront[b];
    const int base = pool.count[b];
    for (int e = tid; e < nf * k; e += blockDim.x) {
      const int fr = e / k, r = e % k;
      const int par = pool.front[b * k + fr];
      const int row = prev.base + b * prev.per_seq + fr;
      pool.score[pb + base + e] = pool.score[pb + par] + (topk_val[(size_t)row * k + r] - lse[row]);
      pool.token[pb + base + e] = topk_idx[(size_t)row * k + r];
      pool.parent[pb + base + e] = par;
      pool.depth[pb + base + e] = t;
      pool.cid[pb + base + e] = (t << 16) | (fr << 8) | r;
      pool.frow[pb + base + e] = -1;
      pool.smask[pb + base + e] = 0ull;
    }
    __syncthreads();
    if (tid == 0) {
      pool.count[b] = base + nf * k;
      s_first = base;
      s_n = nf * k;
    }
  }
  __syncthreads();
  if (t >= depth) return;

  // frontier of depth t: top-k by (score desc, cid asc) among score >= ln tau; else the best one.
  const int first = s_first, ncand = s_n;  // ncand <= k*k <= 256, sorted in two passes of <=128 is not needed:
  // candidates are at most 128 here (k <= 11); larger k uses the same rule over the first 128.
  const int nc = min(ncand, 128);
  for (int i = tid; i < 128; i += blockDim.x) {
    if (i < nc) {
      key[i] = sort_key(pool.score[pb + first + i], pool.cid[pb + first + i]);
      val[i] = first + i;
    } else {
      key[i] = ~0ull;
      val[i] = -1;
    }
  }
  bitonic_sort(key, val, 128);
  __shared__ int s_pass;
  if (tid == 0) {
    int np = 0;
    for (int i = 0; i < nc; ++i)
      if (pool.score[pb + val[i]] >= ln_tau) ++np;
    s_pass = np;
  }
  __syncthreads();
  // Passing candidates are a prefix of the sorted order (score desc), so the
  // frontier is the first min(k, pass) entries, or the single best if none pass.
  const int nf = s_pass > 0 ? min(k, s_pass) : 1;
  for (int i = tid; i < k; i += blockDim.x) {
    const int m = b * k + i;
    if (i < nf) {
      const int e = val[i];
      const int par = pool.parent[pb + e];
      const int sidx = (t - 1) * k + i;
      const uint64_t pm = par < 0 ? 0ull : pool.smask[pb + par];
      const uint64_t sm = pm | (1ull << sidx);
      const int frow = next.base + b * next.per_seq + i;
      pool.front[b * k + i] = e;
      pool.frow[pb + e] = frow;
      pool.smask[pb + e] = sm;
      rows.pos[m] = L + t - 1;
      rows.slot[m] = L + sidx;
      rows.tok[m] = pool.token[pb + e];
      rows.fsrc[m] = par < 0 ? catchup.base + b * catchup.per_seq + c - 1 : pool.frow[pb + par];
      rows.mask[2 * m] = sm;
    } else {
      rows.pos[m] = L;
      rows.slot[m] = -1;
      rows.tok[m] = 0;
      rows.fsrc[m] = catchup.base + b * catchup.per_seq + c - 1;
      rows.mask[2 * m] = 0ull;
    }
    rows.seq[m] = b;
    rows.grp[m] = b;
    rows.mask[2 * m + 1] = 0ull;
  }
  if (tid == 0) {
    pool.nfront[b] = nf;
    Group g;
    g.seq = b;
    g.row0 = b * k;
    g.nrows = k;
    g.prefix = L;
    g.block_len = S;
    groups[b] = g;
  }
}

// n_min > 0: adaptive node count, the candidates whose cumulative confidence
// reaches tau (score >= ln_tau), clamped to [n_min, n_nodes] (reading of the
// 40-120 adaptive count of "EAGLE (LLM decoding)", "EAGLE vs EAGLE-2"); each
// sequence gets its own count, the remaining rows are padding.
__global__ void __launch_bounds__(256) eagle2_final_kernel(State st, Pool pool, int n_nodes, int n_min, float ln_tau,
                                                           TreeOut tree) {
  pdl_wait();
  pdl_trigger();
  __shared__ unsigned long long key[kPoolSort];
  __shared__ int val[kPoolSort];
  __shared__ int tpos[kPoolSort];  // pool index -> tree row (0 = not selected)
  const int b = blockIdx.x, tid = threadIdx.x;
  const size_t pb = (size_t)b * pool.cap;
  const int cnt = min(pool.count[b], kPoolSort);
  int n2 = 1;
  while (n2 < cnt) n2 <<= 1;
  for (int i = tid; i < n2; i += blockDim.x) {
    if (i < cnt) {
      key[i] = sort_key(pool.score[pb + i], pool.cid[pb + i]);
      val[i] = i;
    } else {
      key[i] = ~0ull;
      val[i] = -1;
    }
    tpos[i] = 0;
  }
  bitonic_sort(key, val, n2);
  __shared__ int s_conf;
  if (n_min > 0) {
    if (tid == 0) s_conf = 0;
    __syncthreads();
    int mine = 0;
    for (int i = tid; i < cnt; i += blockDim.x) mine += pool.score[pb + i] >= ln_tau;
    if (mine) atomicAdd(&s_conf, mine);
    __syncthreads();
  }
  const int n = n_min > 0 ? min(min(max(s_conf, n_min), n_nodes), cnt) : min(n_nodes, cnt);
  // re-sort the selected nodes by creation id (depth first): BFS order
  __syncthreads();
  int n3 = 1;
  while (n3 < n) n3 <<= 1;
  for (int i = tid; i < n3; i += blockDim.x) {
    if (i < n) {
      key[i] = (unsigned long long)(unsigned int)pool.cid[pb + val[i]];
    } else {
      key[i] = ~0ull;
      val[i] = -1;
    }
  }
  bitonic_sort(key, val, n3);
  for (int i = tid; i < n; i += blockDim.x) tpos[val[i]] = i + 1;
  __syncthreads();
  const int NR = tree.n_rows;
  if (tid == 0) {
    const int base = b * NR;
    tree.tokens[base] = st.root[b];
    tree.parent[base] = -1;
    tree.depth[base] = 0;
    tree.anc[2 * base] = 1ull;
    tree.anc[2 * base + 1] = 0ull;
    if (tree.score) tree.score[base] = 0.f;
    for (int i = 0; i < NR - 1; ++i) {
      const int j = i + 1, m = base + j;
      if (i < n) {
        const int e = val[i];
        const int par = pool.parent[pb + e];
        const int pj = par < 0 ? 0 : tpos[par];
        tree.tokens[m] = pool.token[pb + e];
        tree.parent[m] = pj;
        tree.depth[m] = pool.depth[pb + e];
        if (tree.score) tree.score[m] = pool.score[pb + e];
        uint64_t a0 = tree.anc[2 * (base + pj)], a1 = tree.anc[2 * (base + pj) + 1];
        if (j < 64) a0 |= 1ull << j; else a1 |= 1ull << (j - 64);
        tree.anc[2 * m] = a0;
        tree.anc[2 * m + 1] = a1;
      } else {
        // padding node: a child of the root with an impossible token, never accepted
        tree.tokens[m] = -1;
        tree.parent[m] = 0;
        tree.depth[m] = 1;
        if (tree.score) tree.score[m] = -INFINITY;
        uint64_t a0 = 1ull, a1 = 0ull;
        if (j < 64) a0 |= 1ull << j; else a1 |= 1ull << (j - 64);
        tree.anc[2 * m] = a0;
        tree.anc[2 * m + 1] = a1;
      }
    }
  }
}

// ---------------------------------------------------------------- accept / commit
__global__ void __launch_bounds__(256) accept_kernel(State st, TreeOut tree, const int* __restrict__ amax,
                                                     const float* __restrict__ h_verify,
                                                     const float* __restrict__ h_low, const float* __restrict__ h_mid,
                                                     int* acc_out, int* tok_out) {
  pdl_wait();
  pdl_trigger();
  __shared__ int path[kMaxDepth + 1];
  __shared__ int s_a, s_bonus, s_over;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int NR = tree.n_rows;
  const int base = b * NR;
  // After any device-detected error (capacity, timeout) the state stops
  // advancing: nothing is committed and nothing is compacted, so no later
  // kernel indexes a slot past the caches.
  if (*(volatile int*)st.status != kStOk) {
    if (tid == 0) {
      st.acc_len[b] = 0;
      if (acc_out) acc_out[b] = -1;
      if (tok_out)
        for (int t = 0; t <= kMaxDepth; ++t) tok_out[b * (kMaxDepth + 1) + t] = -1;
    }
    return;
  }
  if (tid < 32) {
    int cur = 0, a = 0;
    bool over = false;
    if (tid == 0) path[0] = 0;
    for (;;) {
      const int want = amax[base + cur];
      int found = 0x7fffffff;
      for (int j = 1 + tid; j < NR; j += 32)
        if (tree.parent[base + j] == cur && tree.tokens[base + j] == want) found = min(found, j);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) found = min(found, __shfl_xor_sync(0xffffffffu, found, o));
      if (found == 0x7fffffff) break;
      if (a == st.D1 - 1) {  // the accepted path goes on past the catch-up capacity
        over = true;
        break;
      }
      cur = found;
      ++a;
      if (tid == 0) path[a] = cur;
    }
    if (tid == 0) {
      s_a = a;
      s_bonus = amax[base + cur];
      s_over = over;
    }
  }
  __syncthreads();
  if (s_over) {
    if (tid == 0) {
      set_status(st.status, kStInvalid);
      st.acc_len[b] = 0;
      if (acc_out) acc_out[b] = -1;
      if (tok_out)
        for (int t = 0; t <= kMaxDepth; ++t) tok_out[b * (kMaxDepth + 1) + t] = -1;
    }
    return;
  }
  const int a = s_a, bonus = s_bonus;
  const int L = st.L[b];
  // committed features: root and accepted nodes
  for (int e = tid; e < (a + 1) * st.d; e += blockDim.x) {
    const int t = e / st.d, n = e % st.d;
    const size_t dst = ((size_t)b * st.D1 + t) * st.d + n, src = ((size_t)base + path[t]) * st.d + n;
    st.pend_feat[dst] = h_verify[src];
    if (st.pend_low) {
      st.pend_low[dst] = h_low[src];
      st.pend_mid[dst] = h_mid[src];
    }
  }
  if (tid == 0) {
    const int n0 = st.n_out[b];
    for (int t = 0; t <= a; ++t) {
      const int tok = t < a ? tree.tokens[base + path[t + 1]] : bonus;
      st.pend_tok[b * st.D1 + t] = tok;
      if (n0 + t < st.out_cap) st.out[(size_t)b * st.out_cap + n0 + t] = tok;
      st.acc_path[b * st.D1 + t] = path[t];
      if (tok_out) tok_out[b * (kMaxDepth + 1) + t] = tok;
    }
    if (tok_out)
      for (int t = a + 1; t <= kMaxDepth; ++t) tok_out[b * (kMaxDepth + 1) + t] = -1;
    st.n_out[b] = min(n0 + a + 1, st.out_cap);
    st.acc_len[b] = a;
    st.L_prev[b] = L;
    st.L[b] = L + a + 1;
    st.c[b] = a + 1;
    st.root[b] = bonus;
    atomicAdd(&st.hist[a], 1ull);
    if (acc_out) acc_out[b] = a;
  }
}

// Thread i moves dimension i of every accepted row: all reads, then all writes,
// because a destination slot can be another accepted row's source.
template <typename T>
__global__ void compact_kernel(State st, T* kc, T* vc, int n_kv, int hd) {
  pdl_wait();
  pdl_trigger();
  const int l = blockIdx.x, b = blockIdx.y, kvh = blockIdx.z, i = threadIdx.x;
  const int a = st.acc_len[b];
  if (a == 0 || i >= hd) return;
  const int Lp = st.L_prev[b];
  const size_t base = ((((size_t)l * st.B + b) * n_kv + kvh) * st.cap) * hd + i;
  T kk[kMaxDepth], vv[kMaxDepth];
#pragma unroll
  for (int t = 0; t < kMaxDepth; ++t) {
    if (t < a) {
      const size_t src = base + (size_t)(Lp + st.acc_path[b * st.D1 + t + 1]) * hd;
      kk[t] = kc[src];
      vv[t] = vc[src];
    }
  }
#pragma unroll
  for (int t = 0; t < kMaxDepth; ++t) {
    if (t < a) {
      const size_t dst = base + (size_t)(Lp + t + 1) * hd;
      kc[dst] = kk[t];
      vc[dst] = vv[t];
    }
  }
}

__global__ void copy_out_kernel(State st, int max_new, int* d_out) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  for (int i = threadIdx.x; i < max_new; i += blockDim.x)
    d_out[(size_t)b * max_new + i] = i < st.n_out[b] ? st.out[(size_t)b * st.out_cap + i] : -1;
}

}  // namespace

cudaError_t setup_prefill_rows(const int* prompt, int P, int c0, int CL, int B, bool draft, Rows rows,
                               Group* groups, cudaStream_t s) {
  const int n = B * CL;
  return launch_pdl(setup_prefill_kernel, dim3((n + 127) / 128), dim3(128), 0, s, prompt, P, c0, CL, B, draft ? 1 : 0, rows, groups);
}

cudaError_t setup_catchup_rows(State st, Rows rows, Group* groups, cudaStream_t s) {
  return launch_pdl(setup_catchup_kernel, dim3(st.B), dim3(32), 0, s, st, rows, groups);
}

cudaError_t setup_verify_rows(State st, TreeOut tree, Rows rows, Group* groups, Group* groups_local, int spc,
                              cudaStream_t s) {
  return launch_pdl(setup_verify_kernel, dim3(st.B), dim3(128), 0, s, st, tree, rows, groups, groups_local, spc);
}

cudaError_t prefill_finish(State st, const int* root_idx, const float* h_tgt, const float* h_low,
                           const float* h_mid, int CL, int P, int* root_out, cudaStream_t s) {
  return launch_pdl(prefill_finish_kernel, dim3(st.B), dim3(256), 0, s, st, root_idx, h_tgt, h_low, h_mid, CL, P,
                    root_out);
}

cudaError_t set_root_tree(State st, TreeOut tree, cudaStream_t s) {
  return launch_pdl(set_root_tree_kernel, dim3(1), dim3(64), 0, s, st, tree);
}

cudaError_t static_level(State st, StaticTopo topo, int t, const int* topk_idx, const float* topk_val,
                         const float* lse, Level catchup, Level prev, Level next, TreeOut tree, Rows rows,
                         Group* groups, int S, cudaStream_t s) {
  return launch_pdl(static_level_kernel, dim3(st.B), dim3(128), 0, s, st, topo, t, topk_idx, topk_val, lse, catchup,
                    prev, next, tree, rows, groups, S);
}

cudaError_t eagle2_level(State st, Pool pool, int t, int depth, int k, float ln_tau, const int* topk_idx,
                         const float* topk_val, const float* lse, Level catchup, Level prev, Level next,
                         Rows rows, Group* groups, int S, cudaStream_t s) {
  if (k > 11 || k < 1) return cudaErrorInvalidValue;
  return launch_pdl(eagle2_level_kernel, dim3(st.B), dim3(256), 0, s, st, pool, t, depth, k, ln_tau, topk_idx, topk_val, lse, catchup, prev,
                                           next, rows, groups, S);
}

cudaError_t eagle2_final(State st, Pool pool, int n_nodes, int n_min, float ln_tau, TreeOut tree, cudaStream_t s) {
  return launch_pdl(eagle2_final_kernel, dim3(st.B), dim3(256), 0, s, st, pool, n_nodes, n_min, ln_tau, tree);
}

cudaError_t accept_commit(State st, TreeOut tree, const int* amax, const float* h_verify, const float* h_low,
                          const float* h_mid, int* acc_out, int* tok_out, cudaStream_t s) {
  return launch_pdl(accept_kernel, dim3(st.B), dim3(256), 0, s, st, tree, amax, h_verify, h_low, h_mid, acc_out,
                    tok_out);
}

template <typename T>
cudaError_t compact_kv(State st, T* kc, T* vc, int n_layers, int n_kv, int hd, cudaStream_t s) {
  dim3 grid(n_layers, st.B, n_kv);
  return launch_pdl(compact_kernel<T>, dim3(grid), dim3(hd), 0, s, st, kc, vc, n_kv, hd);
}
template cudaError_t compact_kv<float>(State, float*, float*, int, int, int, cudaStream_t);
template cudaError_t compact_kv<__half>(State, __half*, __half*, int, int, int, cudaStream_t);

cudaError_t copy_out(State st, int max_new, int* d_out, cudaStream_t s) {
  return launch_pdl(copy_out_kernel, dim3(st.B), dim3(256), 0, s, st, max_new, d_out);
}

}  // namespace eg
