// Device state of the speculative loop and launchers of the per-step kernels
// (row setup, tree construction, acceptance and compaction).
#pragma once

#include "common.cuh"

namespace eg {

// Per-sequence decoding state, all in device memory so that a whole step can
// be captured in a CUDA graph and replayed without host round trips.
struct State {
  int* L;           // [B] committed KV length
  int* c;           // [B] pending catch-up rows (1 .. D+1)
  int* root;        // [B] x_L: committed, not yet in the KV cache
  int* pend_tok;    // [B][D1] t_{L-c+1} .. t_L
  float* pend_feat; // [B][D1][d] target features f_{L-c} .. f_{L-1}
  float* pend_low;  // fused-feature variant: the low and mid taps of the same rows (NULL otherwise)
  float* pend_mid;
  int* n_out;       // [B] committed tokens
  int* out;         // [B][out_cap]
  int* acc_len;     // [B] accepted draft length of the last commit
  int* acc_path;    // [B][D1] tree rows of the last accepted path (root first)
  int* L_prev;      // [B] L before the last commit
  unsigned long long* hist;  // [kMaxDepth + 1] accepted-length histogram
  int* status;      // device status word
  int B, D1, d, cap, cap_d, out_cap, V;
};

// Static draft-tree topology (BFS order, node 0 = root), device arrays.
struct StaticTopo {
  int n_rows;        // N + 1
  int depth_max;
  int k;             // children per expanded node (max rank + 1)
  const int* parent; // [n_rows]
  const int* rank;   // [n_rows]
  const int* depth;  // [n_rows]
  const int* lrow;   // [n_rows] row of the node's draft forward within its depth level, -1 for leaves
  const int* sidx;   // [n_rows] draft scratch index of non-leaf non-root nodes, -1 otherwise
  const uint64_t* smask;  // [n_rows] scratch-ancestor mask (non-root ancestors and self)
  const int* level_nodes; // [depth_max+1][n_rows] non-leaf nodes per depth, in lrow order
  const int* level_count; // [depth_max+1]
};

// Region of a draft forward inside the draft row buffers: rows [base, base + B * per_seq).
struct Level {
  int base;
  int per_seq;
};

struct TreeOut {
  int n_rows;
  int* tokens;       // [B][n_rows]
  int* parent;
  int* depth;
  uint64_t* anc;     // [B][n_rows][2]
  float* score;      // [B][n_rows] cumulative draft log-confidence (NULL: not tracked)
};

// Dynamic (EAGLE-2) pool, per sequence capacity `cap` entries.
struct Pool {
  float* score;
  int* token;
  int* parent;       // pool index, -1 = root
  int* depth;
  int* cid;          // (depth << 16) | (frontier rank of parent << 8) | child rank
  int* frow;         // row of the node's draft forward (global draft row), -1 if not expanded
  uint64_t* smask;   // scratch-ancestor mask of expanded nodes
  int* count;        // [B]
  int* front;        // [B][k] pool indices of the current frontier
  int* nfront;       // [B]
  int cap;
};

cudaError_t setup_prefill_rows(const int* prompt, int P, int c0, int CL, int B, bool draft, Rows rows,
                               Group* groups, cudaStream_t s);
cudaError_t setup_catchup_rows(State st, Rows rows, Group* groups, cudaStream_t s);
// Also checks the tree (BFS order, parent/depth/ancestor-mask consistency,
// distinct sibling tokens) and records kStInvalid if it is not.
// groups_local[b]: the same group with its rows counted from the first row of
// its verify launch (launches of spc sequences each; spc = 0: one launch).
cudaError_t setup_verify_rows(State st, TreeOut tree, Rows rows, Group* groups, Group* groups_local, int spc,
                              cudaStream_t s);
cudaError_t prefill_finish(State st, const int* root_idx, const float* h_tgt, const float* h_low,
                           const float* h_mid, int CL, int P, int* root_out, cudaStream_t s);
cudaError_t set_root_tree(State st, TreeOut tree, cudaStream_t s);

// Static tree: assign the tokens of depth-t nodes from their parents' top-k
// and, when t < depth_max, write the rows of the depth-t draft forward.
cudaError_t static_level(State st, StaticTopo topo, int t, const int* topk_idx, const float* topk_val,
                         const float* lse, Level catchup, Level prev, Level next, TreeOut tree, Rows rows,
                         Group* groups, int S, cudaStream_t s);

// EAGLE-2: add the children of the frontier expanded at depth t-1 (or of the
// root when t == 1), then, when t < depth, select the depth-t frontier and
// write the rows of its draft forward.
cudaError_t eagle2_level(State st, Pool pool, int t, int depth, int k, float ln_tau, const int* topk_idx,
                         const float* topk_val, const float* lse, Level catchup, Level prev, Level next,
                         Rows rows, Group* groups, int S, cudaStream_t s);
// Top-N of the pool in BFS order -> tree (N = n_nodes, or with n_min > 0 the
// per-sequence adaptive count between n_min and n_nodes; padding rows after).
cudaError_t eagle2_final(State st, Pool pool, int n_nodes, int n_min, float ln_tau, TreeOut tree, cudaStream_t s);

// Greedy accept over the verified tree; commit tokens and features, advance L.
// A path longer than D1 - 1 nodes (only a caller-built tree can hold one) is
// not cut short: nothing is committed and kStInvalid is recorded.
// h_low / h_mid (used when st.pend_low is set): the verify rows' low and mid taps.
cudaError_t accept_commit(State st, TreeOut tree, const int* amax, const float* h_verify, const float* h_low,
                          const float* h_mid, int* acc_out, int* tok_out, cudaStream_t s);
// Move accepted K/V rows to contiguous slots in every layer.
template <typename T>
cudaError_t compact_kv(State st, T* kc, T* vc, int n_layers, int n_kv, int hd, cudaStream_t s);

// Trim committed tokens to max_new per sequence.
cudaError_t copy_out(State st, int max_new, int* d_out, cudaStream_t s);

}  // namespace eg
