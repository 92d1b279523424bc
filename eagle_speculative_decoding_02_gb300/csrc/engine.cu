// Host orchestration of the EAGLE step and the C ABI declared in include/eagle.h.
//
// The context carves one caller-owned workspace into the KV caches, the
// per-phase row buffers and the device-resident decoding state, then enqueues
// each phase as a fixed sequence of kernels on the caller's stream:
//   prefill   target layers over the prompt (chunked), first token, head catch-up
//   draft     head rows for the newly committed positions, then tree expansion
//   verify    target layers over the tree rows, LM-head argmax per row
//   accept    greedy walk, commit, in-place KV compaction
// Shapes never depend on device values, so a step can be captured in a CUDA
// graph and replayed.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/eagle.h"
#include "kernels.h"
#include "stack.h"
#include "step.h"

namespace eg {
namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

struct LayerPtrs {
  const void* wqkv;
  const void* wo;
  const void* wgu;
  const void* wd;
  const float* attn_norm;
  const float* ffn_norm;
  bool w4 = false;  // the four projections are packed int4 blocks (int4.cuh)
};

// Host-derived sizes of a configuration.
// One persistent-kernel program: kind 0 = verify (target layers + LM head),
// kind 1 = draft head forward (FC + head layer + LM head top-k) over M rows
// whose features live at row hbase of the draft buffers.
struct ProgSpec {
  int kind = 0, M = 0, hbase = 0, k = 0;
  int row0 = 0, seq0 = 0, n_seq = 0;            // verify: its rows and sequences (a chunk of the batch)
  int n_phases = 0, n_counters = 0, first = 0;  // first: index of its first phase in the program array
  int first_attn = -1;                          // its first attention phase (set when it is built)
  bool w4 = false;                              // has int4 phases (set when it is built)
};

struct Dims {
  int B = 0, d = 0, Hq = 0, Hkv = 0, hd = 0, ffn = 0, V = 0, Lyr = 0, cap = 0, cap_d = 0, P_max = 0, out_cap = 0;
  int qd = 0, kvd = 0, nqkv = 0;
  int mode = 0, NR = 0, D = 0, D1 = 0, k = 0, S = 0, n_nodes = 0;
  std::vector<int> level_rows;  // rows per sequence of the depth-t draft forward, t = 1..D-1 (index t)
  std::vector<int> level_base;  // absolute first row of level t in the draft buffers (index t)
  int R_d = 0;                      // total draft rows
  int CL = 0;                       // prefill chunk length per sequence
  int M_tgt = 0, M_dft = 0, M_max = 0, M_lm = 0, n_groups_max = 0, ntV = 0, pool_cap = 0;
  bool bf16 = false;
  int verify_spc = 0;               // sequences per verify launch when the batch is split (0: one launch)
  float inv_temp = 0.f;             // 1 / temperature, 0 for greedy decoding
  bool taps = false;                // fused-feature variant: the draft takes fuse [f_low ; f_mid ; f_top]
  int tap_low = 0, tap_mid = 0;     // ... with f_low, f_mid the hidden states after these target layers (1-based)
  int M_fused = 0;                  // rows of the fused-feature buffer
  bool w4 = false;                  // weight-only int4 target projections
  unsigned long long seed = 0;      // sampler seed
  // static topology (host)
  std::vector<int> s_parent, s_rank, s_depth, s_lrow, s_sidx, s_level_nodes, s_level_count;
  std::vector<uint64_t> s_smask, s_anc;
  // Persistent-kernel programs (bf16 models, up to kStackMaxRows rows): the
  // verify pass, and the draft head's forward at catch-up and at every depth.
  std::vector<ProgSpec> progs;
  int stack_M = 0, stack_phases_max = 0, stack_counters_max = 0, stack_phases_total = 0;
};

struct Layout {
  size_t total = 0;
  size_t take(size_t bytes) {
    const size_t at = total;
    total += align_up(bytes);
    return at;
  }
};

}  // namespace
}  // namespace eg

struct eagle_ctx {
  eagle_config cfg{};
  eg::Dims dm;
  cudaStream_t stream = nullptr;
  std::vector<eg::LayerPtrs> layers;
  eg::LayerPtrs head{};
  const void* embed = nullptr;
  const void* lm_head = nullptr;
  const float* final_norm = nullptr;
  const void* fc = nullptr;
  const void* fuse = nullptr;  // fused-feature variant: [d, 3d]
  std::string err;
  bool failed = false;
  int phase = 0;  // 0 fresh, 1 prefilled, 2 drafted, 3 verified
  // buffers
  eg::Rows rows{};
  eg::Group* groups = nullptr;
  eg::Group* groups_local = nullptr;  // verify groups with rows counted from their verify launch's first row
  float* h_tgt = nullptr;
  float* h_dft = nullptr;
  float* h_low = nullptr;   // fused-feature variant: the low / mid taps of the target rows (as h_tgt)
  float* h_mid = nullptr;
  float* fused = nullptr;   // ... and u = fuse [f_low ; f_mid ; f_top] of the rows the draft catches up on
  void* hb = nullptr;
  eg::bf16* hb_lo = nullptr;   // bf16 models: GEMM inputs are hi/lo pairs (x = hb + hb_lo)
  eg::bf16* act_lo = nullptr;
  eg::bf16* attn_lo = nullptr;
  eg::bf16* xfc_lo = nullptr;
  eg::bf16* lm_hb_lo = nullptr;
  float* ssq_a = nullptr;
  float* ssq_b = nullptr;
  void* q = nullptr;
  __half* qg = nullptr;
  void* attn = nullptr;
  void* act = nullptr;
  void* xfc = nullptr;
  void* lm_hb = nullptr;
  float* lm_ssq = nullptr;
  int* lm_src = nullptr;
  float* rec_val = nullptr;
  int* rec_idx = nullptr;
  float* rec_max = nullptr;
  float* rec_sum = nullptr;
  int* dtopk_idx = nullptr;
  float* dtopk_val = nullptr;
  float* dlse = nullptr;
  int* vargmax = nullptr;
  int* root_idx = nullptr;
  eg::TreeOut tree{};
  eg::TreeOut vtree{};  // one-row tree of vanilla decoding
  eg::TreeOut last_tree{};
  eg::State st{};
  eg::Pool pool{};
  eg::StaticTopo topo{};
  float* rope_cos = nullptr;
  float* rope_sin = nullptr;
  void* kc = nullptr;
  void* vc = nullptr;
  void* kc_d = nullptr;
  void* vc_d = nullptr;
  void* gemm_scratch = nullptr;
  size_t gemm_scratch_bytes = 0;
  void* w4_dense = nullptr;  // int4 targets, per-operation path: the current projection expanded to dtype
  float* attn_part = nullptr;
  eg::StackPhase* stack_prog = nullptr;  // every program's phases, back to back
  void* stack_scratch = nullptr;
  float* stack_part = nullptr;
  unsigned long long* trace = nullptr;   // caller's phase-trace buffer (eagle_set_trace)
  cudaGraphExec_t graph_exec[2] = {nullptr, nullptr};  // captured step: [0] speculative, [1] vanilla
  int graph_kernels[2] = {-1, -1};                       // kernel nodes in each captured step
};

namespace eg {
namespace {

eagle_status fail(eagle_ctx* c, eagle_status s, const std::string& msg) {
  if (c) {
    c->err = msg;
    if (s != EAGLE_ERR_INVALID_ARG) c->failed = true;
  }
  return s;
}

#define EG_CK(call)                                                                             \
  do {                                                                                          \
    cudaError_t e_ = (call);                                                                    \
    if (e_ != cudaSuccess)                                                                      \
      return fail(c, EAGLE_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_));      \
  } while (0)

#define EG_TRY(call)                   \
  do {                                 \
    eagle_status s_ = (call);          \
    if (s_ != EAGLE_OK) return s_;     \
  } while (0)

bool gemm_tc_ok(const Dims& dm, int N, int K) {
  return dm.bf16 && N % kTileN == 0 && K % 64 == 0;
}

eagle_status derive(const eagle_config& cfg, Dims& dm, std::string& why) {
  auto bad = [&](const char* m) { why = m; return EAGLE_ERR_INVALID_ARG; };
  if (cfg.n_layers <= 0 || cfg.d <= 0 || cfg.n_heads <= 0 || cfg.n_kv_heads <= 0 || cfg.ffn <= 0 ||
      cfg.vocab <= 0 || cfg.batch <= 0 || cfg.kv_cap <= 0 || cfg.max_prompt <= 0 || cfg.max_new <= 0)
    return bad("non-positive dimension");
  if (cfg.dtype != EAGLE_DTYPE_F32 && cfg.dtype != EAGLE_DTYPE_BF16) return bad("dtype");
  if (cfg.d % kTileN) { why = "d must be a multiple of 128"; return EAGLE_ERR_UNSUPPORTED; }
  if (cfg.head_dim != 64 && cfg.head_dim != 128) { why = "head_dim must be 64 or 128"; return EAGLE_ERR_UNSUPPORTED; }
  if (cfg.n_heads % cfg.n_kv_heads) return bad("n_kv_heads must divide n_heads");
  if (!(cfg.rms_eps > 0.f) || !(cfg.rope_theta > 0.f)) return bad("rms_eps / rope_theta");
  if (!(cfg.temperature >= 0.f) || !std::isfinite(cfg.temperature)) return bad("temperature must be finite, >= 0");
  dm.inv_temp = cfg.temperature > 0.f ? 1.f / cfg.temperature : 0.f;
  dm.seed = cfg.seed;
  dm.B = cfg.batch; dm.d = cfg.d; dm.Hq = cfg.n_heads; dm.Hkv = cfg.n_kv_heads; dm.hd = cfg.head_dim;
  dm.ffn = cfg.ffn; dm.V = cfg.vocab; dm.Lyr = cfg.n_layers; dm.cap = cfg.kv_cap; dm.P_max = cfg.max_prompt;
  dm.qd = dm.Hq * dm.hd; dm.kvd = dm.Hkv * dm.hd; dm.nqkv = dm.qd + 2 * dm.kvd;
  dm.bf16 = cfg.dtype == EAGLE_DTYPE_BF16;
  if (dm.bf16 && (dm.ffn % 64)) { why = "bf16 models need ffn % 64 == 0"; return EAGLE_ERR_UNSUPPORTED; }
  dm.mode = cfg.tree_mode;
  dm.n_nodes = cfg.n_nodes;
  if (cfg.n_nodes < 1 || cfg.n_nodes + 1 > kMaxTreeRows) return bad("n_nodes must be in 1..120");
  if (cfg.feature_taps != 0 && cfg.feature_taps != 1 && cfg.feature_taps != 3) return bad("feature_taps must be 0, 1 or 3");
  dm.taps = cfg.feature_taps == 3;
  if (cfg.weight_bits != 0 && cfg.weight_bits != 16 && cfg.weight_bits != 4) return bad("weight_bits must be 0, 16 or 4");
  dm.w4 = cfg.weight_bits == 4;
  if (dm.w4 && (cfg.d % 64 || (cfg.n_heads * cfg.head_dim) % 64 || cfg.ffn % 64 ||
                ((cfg.n_heads + 2 * cfg.n_kv_heads) * cfg.head_dim) % 128)) {
    why = "int4 weights need d, n_heads * head_dim and ffn to be multiples of 64";
    return EAGLE_ERR_UNSUPPORTED;
  }
  dm.tap_low = std::max(1, dm.taps ? cfg.n_layers / 4 : 0);
  dm.tap_mid = std::max(1, dm.taps ? cfg.n_layers / 2 : 0);
  dm.NR = cfg.n_nodes + 1;
  dm.level_rows.assign(kMaxDepth + 1, 0);
  dm.level_base.assign(kMaxDepth + 1, 0);
  if (cfg.tree_mode == EAGLE_TREE_STATIC) {
    if (!cfg.static_parent || !cfg.static_rank) return bad("static tree arrays missing");
    const int NR = dm.NR;
    dm.s_parent.assign(cfg.static_parent, cfg.static_parent + NR);
    dm.s_rank.assign(cfg.static_rank, cfg.static_rank + NR);
    if (dm.s_parent[0] != -1) return bad("static_parent[0] must be -1");
    dm.s_depth.assign(NR, 0);
    int kmax = 0, D = 0;
    for (int j = 1; j < NR; ++j) {
      const int p = dm.s_parent[j];
      if (p < 0 || p >= j) return bad("static tree must be in BFS order (0 <= parent[j] < j)");
      if (dm.s_rank[j] < 0 || dm.s_rank[j] >= kMaxTopK) return bad("static rank out of range");
      dm.s_depth[j] = dm.s_depth[p] + 1;
      if (j > 1 && dm.s_depth[j] < dm.s_depth[j - 1]) return bad("static tree must be in BFS order (depth)");
      for (int i = 1; i < j; ++i)
        if (dm.s_parent[i] == p && dm.s_rank[i] == dm.s_rank[j]) return bad("duplicate sibling rank");
      kmax = std::max(kmax, dm.s_rank[j] + 1);
      D = std::max(D, dm.s_depth[j]);
    }
    if (D > kMaxDepth) return bad("static tree deeper than 8");
    dm.D = D; dm.k = kmax;
    std::vector<int> has_kids(NR, 0);
    for (int j = 1; j < NR; ++j) has_kids[dm.s_parent[j]] = 1;
    dm.s_lrow.assign(NR, -1); dm.s_sidx.assign(NR, -1); dm.s_smask.assign(NR, 0);
    dm.s_level_nodes.assign((size_t)(D + 1) * NR, 0); dm.s_level_count.assign(D + 1, 0);
    int S = 0;
    for (int j = 1; j < NR; ++j) {
      if (!has_kids[j]) continue;
      const int t = dm.s_depth[j];
      dm.s_lrow[j] = dm.s_level_count[t];
      dm.s_level_nodes[(size_t)t * NR + dm.s_level_count[t]] = j;
      dm.s_level_count[t]++;
      dm.s_sidx[j] = S++;
    }
    if (S > 64) return bad("static tree has more than 64 expanded nodes");
    for (int j = 1; j < NR; ++j) {
      if (!has_kids[j]) continue;
      uint64_t m = 0;
      for (int a = j; a > 0; a = dm.s_parent[a]) m |= 1ull << dm.s_sidx[a];
      dm.s_smask[j] = m;
    }
    dm.S = S;
    for (int t = 1; t < D; ++t) dm.level_rows[t] = dm.s_level_count[t];
    dm.s_anc.assign((size_t)NR * 2, 0);
    for (int j = 0; j < NR; ++j)
      for (int a = j; a >= 0; a = a ? dm.s_parent[a] : -1) {
        dm.s_anc[2 * j + a / 64] |= 1ull << (a % 64);
        if (a == 0) break;
      }
    if (cfg.n_nodes_min != 0) return bad("n_nodes_min applies to dynamic trees only");
  } else if (cfg.tree_mode == EAGLE_TREE_DYNAMIC) {
    if (cfg.top_k < 1 || cfg.top_k > 11) return bad("top_k must be in 1..11");
    if (cfg.depth < 1 || cfg.depth > kMaxDepth) return bad("depth must be in 1..8");
    if (!(cfg.tau > 0.f) || cfg.tau > 1.f) return bad("tau must be in (0, 1]");
    dm.D = cfg.depth; dm.k = cfg.top_k;
    dm.S = (dm.D - 1) * dm.k;
    if (dm.S > 64) return bad("(depth-1)*top_k must be <= 64");
    for (int t = 1; t < dm.D; ++t) dm.level_rows[t] = dm.k;
    dm.pool_cap = dm.k + (dm.D - 1) * dm.k * dm.k;
    if (dm.pool_cap > 1024) return bad("pool larger than 1024");
    if (dm.pool_cap < dm.n_nodes) return bad("n_nodes exceeds the candidate pool");
    if (cfg.n_nodes_min < 0 || cfg.n_nodes_min > cfg.n_nodes) return bad("n_nodes_min must be in 0..n_nodes");
  } else {
    return bad("tree_mode");
  }
  dm.D1 = dm.D + 1;
  int base = dm.B * dm.D1;
  for (int t = 1; t < dm.D; ++t) {
    dm.level_base[t] = base;
    base += dm.B * dm.level_rows[t];
  }
  dm.R_d = base;
  dm.cap_d = (dm.cap + dm.S + 7) / 8 * 8;
  dm.out_cap = cfg.max_new + dm.D1 + 1;
  const int rows_budget = 8192;
  int CL = std::max(128, rows_budget / dm.B / 128 * 128);
  dm.CL = std::min(dm.P_max, CL);
  const int M_pf = dm.B * dm.CL;
  dm.M_tgt = std::max(dm.B * kMaxTreeRows, M_pf);
  dm.M_dft = std::max(dm.R_d, M_pf);
  dm.M_max = std::max(dm.M_tgt, dm.M_dft);
  dm.M_fused = dm.taps ? std::max(M_pf, dm.B * dm.D1) : 0;
  int lvl_max = dm.D1;
  for (int t = 1; t < dm.D; ++t) lvl_max = std::max(lvl_max, dm.level_rows[t]);
  dm.M_lm = std::max(dm.B * kMaxTreeRows, dm.B * lvl_max);
  dm.n_groups_max = std::max(dm.B * ((dm.CL + 127) / 128), dm.B);
  dm.ntV = (dm.V + kTileN - 1) / kTileN;
  if (dm.P_max + cfg.max_new + dm.D1 + dm.NR > dm.cap) {
    why = "kv_cap too small for max_prompt + max_new + tree";
    return EAGLE_ERR_INVALID_ARG;
  }
  if (dm.bf16 && dm.nqkv % kTileN == 0 && dm.qd % 64 == 0 && dm.V % kTileN == 0) {
    const int layer_tiles = dm.nqkv / kTileN + dm.d / kTileN + 2 * dm.ffn / kTileN + dm.d / kTileN;
    auto add = [&](int kind, int M, int hbase, int k) {
      if (!stack_supported(M, dm.hd)) return;
      ProgSpec p;
      p.kind = kind; p.M = M; p.hbase = hbase; p.k = k;
      const int layers = kind == 0 ? dm.Lyr : 1;
      p.n_phases = 6 * layers + 1 + (kind == 1 ? 1 : 0);  // per layer: QKV, attention, merge, O, gate/up, down
      p.n_counters = layers * layer_tiles + dm.ntV + (kind == 1 ? dm.d / kTileN : 0);
      p.first = dm.stack_phases_total;
      dm.stack_phases_total += p.n_phases;
      dm.stack_M = std::max(dm.stack_M, M);
      dm.stack_phases_max = std::max(dm.stack_phases_max, p.n_phases);
      dm.stack_counters_max = std::max(dm.stack_counters_max, p.n_counters);
      dm.progs.push_back(p);
    };
    if (stack_supported(dm.B * dm.NR, dm.hd)) {
      add(0, dm.B * dm.NR, 0, 1);
      if (!dm.progs.empty()) dm.progs.back().n_seq = dm.B;
    } else if (stack_supported(dm.NR, dm.hd) &&
               (dm.B + kStackMaxRows / dm.NR - 1) / (kStackMaxRows / dm.NR) <= 2) {
      // more tree rows than one launch takes: two launches over halves of the
      // batch (whole sequences), each streaming the weights once. (Measured at 61-row
      // trees: batch 4 verify 17.1 -> 14.4 ms against the per-operation kernels; at
      // batch 16 eight such launches, 7.2 ms each at 122 rows where the hi/lo pairs
      // make the tensor work equal the weight stream, lose to them: 57.8 vs 54 ms.)
      dm.verify_spc = kStackMaxRows / dm.NR;
      for (int s0 = 0; s0 < dm.B; s0 += dm.verify_spc) {
        const int ns = std::min(dm.verify_spc, dm.B - s0);
        add(0, ns * dm.NR, 0, 1);
        ProgSpec& p = dm.progs.back();
        p.row0 = s0 * dm.NR;
        p.seq0 = s0;
        p.n_seq = ns;
      }
    }
    add(1, dm.B * dm.D1, 0, dm.k);
    for (int t = 1; t < dm.D; ++t)
      if (dm.level_rows[t] > 0) add(1, dm.B * dm.level_rows[t], dm.level_base[t], dm.k);
  }
  return EAGLE_OK;
}

struct Offsets {
  size_t rows_seq, rows_pos, rows_slot, rows_grp, rows_tok, rows_fsrc, rows_mask, groups, groups_local;
  size_t h_tgt, h_dft, h_low, h_mid, fused, hb, ssq_a, ssq_b, q, qg, attn, act, xfc, lm_hb, lm_ssq, lm_src;
  size_t hb_lo, act_lo, attn_lo, xfc_lo, lm_hb_lo;
  size_t rec_val, rec_idx, rec_max, rec_sum, dtopk_idx, dtopk_val, dlse, vargmax, root_idx;
  size_t t_tok, t_par, t_dep, t_anc, t_score, vt_tok, vt_par, vt_dep, vt_anc;
  size_t L, c, root, pend_tok, pend_feat, pend_low, pend_mid, n_out, out, acc_len, acc_path, L_prev, hist, status;
  size_t p_score, p_token, p_parent, p_depth, p_cid, p_frow, p_smask, p_count, p_front, p_nfront;
  size_t s_parent, s_rank, s_depth, s_lrow, s_sidx, s_smask, s_lnodes, s_lcount;
  size_t rope_cos, rope_sin, kc, vc, kc_d, vc_d, gemm, attn_part, stack_prog, stack_scratch, stack_part, w4_dense;
  size_t gemm_bytes;
  size_t total;
};

Offsets plan(const Dims& dm) {
  Offsets o{};
  Layout L;
  const size_t es = dm.bf16 ? 2 : 4;
  const size_t M = dm.M_max;
  const int nt_d = dm.d / kTileN;
  o.rows_seq = L.take(M * 4); o.rows_pos = L.take(M * 4); o.rows_slot = L.take(M * 4);
  o.rows_grp = L.take(M * 4); o.rows_tok = L.take(M * 4); o.rows_fsrc = L.take(M * 4);
  o.rows_mask = L.take(M * 16); o.groups = L.take((size_t)dm.n_groups_max * sizeof(Group));
  o.groups_local = L.take((size_t)dm.B * sizeof(Group));
  o.h_tgt = L.take((size_t)dm.M_tgt * dm.d * 4);
  o.h_dft = L.take((size_t)dm.M_dft * dm.d * 4);
  const size_t tap_rows = dm.taps ? dm.M_tgt : 0;
  o.h_low = L.take(tap_rows * dm.d * 4); o.h_mid = L.take(tap_rows * dm.d * 4);
  o.fused = L.take((size_t)dm.M_fused * dm.d * 4);
  const int xw = dm.taps ? 3 : 2;  // width of the FC / fuse GEMM input, in units of d
  o.hb = L.take(M * dm.d * es);
  o.ssq_a = L.take(M * nt_d * 4); o.ssq_b = L.take(M * nt_d * 4);
  o.q = L.take(M * dm.qd * 4); o.qg = L.take(M * dm.qd * 2); o.attn = L.take(M * dm.qd * es);
  o.act = L.take(M * dm.ffn * es); o.xfc = L.take(M * xw * dm.d * es);
  o.lm_hb = L.take((size_t)dm.B * dm.d * es); o.lm_ssq = L.take((size_t)dm.B * nt_d * 4);
  const size_t lo = dm.bf16 ? 2 : 0;  // low halves of the hi/lo GEMM inputs (bf16 models only)
  o.hb_lo = L.take(M * dm.d * lo); o.act_lo = L.take(M * dm.ffn * lo); o.attn_lo = L.take(M * dm.qd * lo);
  o.xfc_lo = L.take(M * xw * dm.d * lo); o.lm_hb_lo = L.take((size_t)dm.B * dm.d * lo);
  o.lm_src = L.take((size_t)dm.B * 4);
  const size_t nrec = (size_t)dm.ntV * dm.M_lm;
  const int krec = std::max(dm.k, 1);
  o.rec_val = L.take(nrec * krec * 4); o.rec_idx = L.take(nrec * krec * 4);
  o.rec_max = L.take(nrec * 4); o.rec_sum = L.take(nrec * 4);
  o.dtopk_idx = L.take((size_t)dm.R_d * krec * 4); o.dtopk_val = L.take((size_t)dm.R_d * krec * 4);
  o.dlse = L.take((size_t)dm.R_d * 4);
  o.vargmax = L.take((size_t)dm.B * kMaxTreeRows * 4); o.root_idx = L.take((size_t)dm.B * 4);
  const size_t tn = (size_t)dm.B * kMaxTreeRows;
  o.t_tok = L.take(tn * 4); o.t_par = L.take(tn * 4); o.t_dep = L.take(tn * 4); o.t_anc = L.take(tn * 16);
  o.t_score = L.take(tn * 4);
  o.vt_tok = L.take(dm.B * 4); o.vt_par = L.take(dm.B * 4); o.vt_dep = L.take(dm.B * 4); o.vt_anc = L.take(dm.B * 16);
  const size_t B = dm.B;
  o.L = L.take(B * 4); o.c = L.take(B * 4); o.root = L.take(B * 4);
  o.pend_tok = L.take(B * dm.D1 * 4); o.pend_feat = L.take(B * dm.D1 * dm.d * 4);
  o.pend_low = L.take(dm.taps ? B * dm.D1 * dm.d * 4 : 0); o.pend_mid = L.take(dm.taps ? B * dm.D1 * dm.d * 4 : 0);
  o.n_out = L.take(B * 4); o.out = L.take(B * dm.out_cap * 4); o.acc_len = L.take(B * 4);
  o.acc_path = L.take(B * dm.D1 * 4); o.L_prev = L.take(B * 4);
  o.hist = L.take((kMaxDepth + 1) * 8); o.status = L.take(4);
  const size_t pc = (size_t)std::max(dm.pool_cap, 1) * B;
  o.p_score = L.take(pc * 4); o.p_token = L.take(pc * 4); o.p_parent = L.take(pc * 4); o.p_depth = L.take(pc * 4);
  o.p_cid = L.take(pc * 4); o.p_frow = L.take(pc * 4); o.p_smask = L.take(pc * 8);
  o.p_count = L.take(B * 4); o.p_front = L.take(B * std::max(dm.k, 1) * 4); o.p_nfront = L.take(B * 4);
  const size_t NR = dm.NR;
  o.s_parent = L.take(NR * 4); o.s_rank = L.take(NR * 4); o.s_depth = L.take(NR * 4); o.s_lrow = L.take(NR * 4);
  o.s_sidx = L.take(NR * 4); o.s_smask = L.take(NR * 8); o.s_lnodes = L.take((dm.D + 1) * NR * 4);
  o.s_lcount = L.take((dm.D + 1) * 4);
  o.rope_cos = L.take((size_t)dm.cap_d * (dm.hd / 2) * 4); o.rope_sin = L.take((size_t)dm.cap_d * (dm.hd / 2) * 4);
  const size_t kvl = B * dm.Hkv * (size_t)dm.cap * dm.hd * es;
  o.kc = L.take(kvl * dm.Lyr); o.vc = L.take(kvl * dm.Lyr);
  const size_t kvd = B * dm.Hkv * (size_t)dm.cap_d * dm.hd * es;
  o.kc_d = L.take(kvd); o.vc_d = L.take(kvd);
  size_t g = 0;
  if (dm.bf16) {
    const int Ns[] = {dm.nqkv, dm.d, 2 * dm.ffn, dm.d, dm.V};
    const int Ks[] = {dm.d, dm.qd, dm.d, dm.ffn, dm.d};
    for (int i = 0; i < 5; ++i) g = std::max(g, gemm_tc_scratch_bytes((int)M, Ns[i], Ks[i]));
    g = std::max(g, gemm_tc_scratch_bytes((int)M, dm.d, xw * dm.d));
  }
  o.gemm_bytes = g;
  o.gemm = L.take(std::max<size_t>(g, 256));
  size_t wmax = 0;  // largest target projection, expanded (int4 targets)
  if (dm.w4) {
    const size_t Ns[] = {(size_t)dm.nqkv, (size_t)dm.d, 2 * (size_t)dm.ffn, (size_t)dm.d};
    const size_t Ks[] = {(size_t)dm.d, (size_t)dm.qd, (size_t)dm.d, (size_t)dm.ffn};
    for (int i = 0; i < 4; ++i) wmax = std::max(wmax, Ns[i] * Ks[i] * es);
  }
  o.w4_dense = L.take(wmax);
  o.attn_part = L.take(std::max<size_t>(
      dm.bf16 ? attention_umma_part_bytes((int)M, dm.Hq, dm.Hkv, dm.hd, dm.cap_d) : 0,
      256));
  o.stack_prog = L.take((size_t)dm.stack_phases_total * sizeof(StackPhase));
  o.stack_scratch = L.take(dm.progs.empty() ? 0 : stack_scratch_bytes(dm.stack_M, dm.stack_phases_max,
                                                                          dm.stack_counters_max));
  o.stack_part = L.take(dm.progs.empty() ? 0 : stack_attention_part_bytes(dm.stack_M, dm.Hq, dm.Hkv, dm.hd, dm.cap_d));
  o.total = L.total;
  return o;
}

template <typename T>
struct Eng {
  static eagle_status gemm(eagle_ctx* c, const void* X, const bf16* X_lo, const void* W, int M, int N, int K,
                           const EpiParams& ep, bool w_dep = false) {
    if (M <= 0) return EAGLE_OK;
    if constexpr (sizeof(T) == 2) {
      if (gemm_tc_ok(c->dm, N, K)) {
        EG_CK(gemm_tc((const bf16*)X, X_lo, (const bf16*)W, M, N, K, ep, c->gemm_scratch, c->st.status, c->stream,
                      w_dep));
        return EAGLE_OK;
      }
    }
    EG_CK(gemm_simt<T>((const T*)X, (const T*)W, M, N, K, ep, c->stream));
    return EAGLE_OK;
  }

  static eagle_status attention(eagle_ctx* c, const AttnArgs& a) {
    if constexpr (sizeof(T) == 2) {
      EG_CK(attention_umma(a, c->stream));
    } else {
      EG_CK(attention_simt<T>(a, c->stream));
    }
    return EAGLE_OK;
  }

  // Low halves of the hi/lo activation pairs: bf16 models carry every GEMM and
  // attention activation as a hi/lo bf16 pair (about float32 precision at no
  // HBM cost: the weights set the bytes). Weight-only int4 models do not
  // (W4A16: bf16 activations): their 4-bit weights err far more than a bf16
  // activation does, so the pairs' second operand bought no accuracy there and
  // cost MMA work and ring space (8B int4 verify 5.78 -> 5.53 ms without it).
  static bool pairs(const eagle_ctx* c) { return sizeof(T) == 2 && !c->dm.w4; }
  static bf16* lo(const eagle_ctx* c, bf16* p) { return pairs(c) ? p : nullptr; }

  static EpiParams epi(eagle_ctx* c, int kind, int M, int N) {
    EpiParams e;
    e.kind = kind;
    e.M = M;
    e.N = N;
    e.eps = c->cfg.rms_eps;
    return e;
  }

  // Sinks of a forward phase's op sequence: Direct runs each op as its own
  // kernel(s); Record appends it to a persistent-kernel program.
  struct Direct {
    eagle_ctx* c;
    eagle_status gemm(const void* X, const bf16* X_lo, const void* W, int M, int N, int K, const EpiParams& e,
                      bool w4 = false) {
      if (w4) {  // expand the int4 projection, then the dense GEMM (which must wait for it before its weights)
        if (M <= 0) return EAGLE_OK;
        EG_CK(int4_dequant<T>(W, N, K, (T*)c->w4_dense, c->stream));
        return Eng::gemm(c, X, X_lo, c->w4_dense, M, N, K, e, true);
      }
      return Eng::gemm(c, X, X_lo, W, M, N, K, e);
    }
    eagle_status attention(const AttnArgs& a) { return Eng::attention(c, a); }
  };
  struct Record {
    eagle_ctx* c;
    StackProgramBuilder* b;
    eagle_status gemm(const void* X, const bf16* X_lo, const void* W, int M, int N, int K, const EpiParams& e,
                      bool w4 = false) {
      (void)M;
      StackGemmDesc g{(const bf16*)W, (const bf16*)X, X_lo, c->dm.M_max, N, K, e, w4};
      b->gemm(g);
      return b->ok ? EAGLE_OK : fail(c, EAGLE_ERR_UNSUPPORTED, "persistent program: GEMM shape");
    }
    eagle_status attention(const AttnArgs& a) {
      AttnArgs r = a;
      r.part = c->stack_part;
      b->attention(r);
      return EAGLE_OK;
    }
  };

  // One pre-norm decoder layer over M rows whose (hb, ssq_b) hold the layer input.
  // Per-row metadata of rows [row0, ...) (a verify launch over a chunk of the batch).
  static Rows rows_at(const Rows& r, int row0) {
    return Rows{r.seq + row0, r.pos + row0, r.slot + row0, r.grp + row0, r.mask + 2 * row0, r.tok + row0,
                r.fsrc + row0};
  }

  // rows of the layer: M rows from row row0 of the metadata (their residual stream
  // at h), attention groups `groups` (NULL: c->groups); the GEMM inputs and the
  // other intermediates are the row buffers from their first row.
  template <typename Sink>
  static eagle_status layer(eagle_ctx* c, Sink& sink, const LayerPtrs& lw, void* kc, void* vc, int cap, int M,
                            int n_groups, float* h, const float* gain_next, int row0 = 0,
                            const Group* groups = nullptr, float* tap = nullptr, float* tap2 = nullptr) {
    const Dims& dm = c->dm;
    const Rows rows = rows_at(c->rows, row0);
    EpiParams e = epi(c, kEpiQkv, M, dm.nqkv);
    e.ssq_in = c->ssq_b; e.n_ssq_in = dm.d / kTileN; e.inv_d_in = 1.f / dm.d;
    // float32 queries only for the SIMT attention of float32 models; the tcgen05
    // attention of bf16 models reads the grouped half queries
    e.out = sizeof(T) == 2 ? nullptr : c->q; e.q_dim = dm.qd; e.kv_dim = dm.kvd; e.head_dim = dm.hd; e.n_kv = dm.Hkv; e.cap = cap;
    const float scale = 1.f / std::sqrt((float)dm.hd);
    e.qg = c->qg; e.qg_scale = scale * 1.4426950408889634f;
    e.rope_cos = c->rope_cos; e.rope_sin = c->rope_sin; e.kc = kc; e.vc = vc; e.rows = rows;
    EG_TRY(sink.gemm(c->hb, lo(c, c->hb_lo), lw.wqkv, M, dm.nqkv, dm.d, e, lw.w4));

    AttnArgs a{};
    a.q = (const float*)c->q; a.qg = c->qg; a.kc = kc; a.vc = vc; a.o = c->attn; a.o_lo = lo(c, c->attn_lo);
    a.groups = groups ? groups : c->groups; a.n_groups = n_groups;
    a.mask = rows.mask; a.row_grp = rows.grp; a.M = M; a.Hq = dm.Hq; a.Hkv = dm.Hkv; a.hd = dm.hd; a.cap = cap; a.n_seq = dm.B;
    a.max_prefix = cap; a.scale = scale; a.part = c->attn_part; a.status = c->st.status;
    EG_TRY(sink.attention(a));

    e = epi(c, kEpiResid, M, dm.d);
    e.h = h; e.hb = c->hb; e.hb_lo = lo(c, c->hb_lo); e.ssq_out = c->ssq_a; e.gain = lw.ffn_norm;
    EG_TRY(sink.gemm(c->attn, lo(c, c->attn_lo), lw.wo, M, dm.d, dm.qd, e, lw.w4));

    e = epi(c, kEpiSwiglu, M, 2 * dm.ffn);
    e.ssq_in = c->ssq_a; e.n_ssq_in = dm.d / kTileN; e.inv_d_in = 1.f / dm.d; e.out = c->act; e.ffn = dm.ffn;
    e.out_lo = lo(c, c->act_lo);
    EG_TRY(sink.gemm(c->hb, lo(c, c->hb_lo), lw.wgu, M, 2 * dm.ffn, dm.d, e, lw.w4));

    e = epi(c, kEpiResid, M, dm.d);
    e.h = h; e.hb = c->hb; e.hb_lo = lo(c, c->hb_lo); e.ssq_out = c->ssq_b; e.gain = gain_next;
    e.h_tap = tap; e.h_tap2 = tap2;
    EG_TRY(sink.gemm(c->act, lo(c, c->act_lo), lw.wd, M, dm.d, dm.ffn, e, lw.w4));
    return EAGLE_OK;
  }

  // LM-head GEMM with per-tile top-k records (merged by lm_head_merge). choose:
  // the rows pick the target's next token (verify, prefill), so at T > 0 the
  // records are of the Gumbel-perturbed logits (the sample); the rows' positions
  // and sequences are in c->rows, through idx (row -> rows entry) when not NULL.
  template <typename Sink>
  static eagle_status lm_head_gemm(eagle_ctx* c, Sink& sink, const void* X, const bf16* X_lo, const float* ssq,
                                   int M, int k, float* logits, bool choose = false, const int* idx = nullptr,
                                   int row0 = 0) {
    const Dims& dm = c->dm;
    EpiParams e = epi(c, kEpiLmHead, M, dm.V);
    e.ssq_in = ssq; e.n_ssq_in = dm.d / kTileN; e.inv_d_in = 1.f / dm.d; e.topk = k; e.y = logits;
    e.rec_val = c->rec_val; e.rec_idx = c->rec_idx; e.rec_max = c->rec_max; e.rec_sum = c->rec_sum;
    if (choose && dm.inv_temp > 0.f) {
      e.inv_temp = dm.inv_temp; e.seed = dm.seed;
      e.samp_pos = c->rows.pos + row0; e.samp_seq = c->rows.seq + row0; e.samp_idx = idx;
    }
    return sink.gemm(X, X_lo, c->lm_head, M, dm.V, dm.d, e);
  }

  static eagle_status lm_head_merge(eagle_ctx* c, int M, int k, int* idx, float* val, float* lse) {
    EG_CK(topk_merge(c->rec_val, c->rec_idx, c->rec_max, c->rec_sum, c->dm.ntV, M, k, idx, val, lse, c->stream));
    return EAGLE_OK;
  }

  static eagle_status lm_head(eagle_ctx* c, const void* X, const bf16* X_lo, const float* ssq, int M, int k,
                              int* idx, float* val, float* lse, float* logits, bool choose = false,
                              const int* rows_idx = nullptr) {
    Direct d{c};
    EG_TRY(lm_head_gemm(c, d, X, X_lo, ssq, M, k, logits, choose, rows_idx));
    return lm_head_merge(c, M, k, idx, val, lse);
  }

  template <typename Sink>
  static eagle_status target_layers(eagle_ctx* c, Sink& sink, int M, int n_groups, int row0 = 0,
                                    const Group* groups = nullptr) {
    const Dims& dm = c->dm;
    const size_t kvl = (size_t)dm.B * dm.Hkv * dm.cap * dm.hd * sizeof(T);
    for (int l = 0; l < dm.Lyr; ++l) {
      const float* gn = l + 1 < dm.Lyr ? c->layers[l + 1].attn_norm : c->final_norm;
      // fused-feature variant: the hidden states after the tap layers are copied out
      float* t1 = dm.taps && l + 1 == dm.tap_low ? c->h_low + (size_t)row0 * dm.d : nullptr;
      float* t2 = dm.taps && l + 1 == dm.tap_mid ? c->h_mid + (size_t)row0 * dm.d : nullptr;
      EG_TRY(layer(c, sink, c->layers[l], (char*)c->kc + l * kvl, (char*)c->vc + l * kvl, dm.cap, M, n_groups,
                   c->h_tgt + (size_t)row0 * dm.d, gn, row0, groups, t1, t2));
    }
    return EAGLE_OK;
  }

  static eagle_status embed(eagle_ctx* c, int M, int row0 = 0) {
    const Dims& dm = c->dm;
    EG_CK(embed_rows<T>((const T*)c->embed, c->rows.tok + row0, M, dm.d, c->layers[0].attn_norm,
                        c->h_tgt + (size_t)row0 * dm.d, (T*)c->hb, lo(c, c->hb_lo), c->ssq_b, c->stream));
    return EAGLE_OK;
  }

  static eagle_status target_stack(eagle_ctx* c, int M, int n_groups) {
    Direct d{c};
    EG_TRY(embed(c, M));
    return target_layers(c, d, M, n_groups);
  }

  // FC([feature ; E(token)]) -> head layer -> (k > 0) LM head, over rows whose features sit at row hbase.
  template <typename Sink>
  static eagle_status draft_ops(eagle_ctx* c, Sink& sink, int M, int n_groups, int hbase, int k) {
    const Dims& dm = c->dm;
    float* h = c->h_dft + (size_t)hbase * dm.d;
    EpiParams e = epi(c, kEpiFc, M, dm.d);
    e.h = h; e.hb = c->hb; e.hb_lo = lo(c, c->hb_lo); e.ssq_out = c->ssq_b; e.gain = c->head.attn_norm;
    EG_TRY(sink.gemm(c->xfc, lo(c, c->xfc_lo), c->fc, M, dm.d, 2 * dm.d, e));
    EG_TRY(layer(c, sink, c->head, c->kc_d, c->vc_d, dm.cap_d, M, n_groups, h, c->final_norm));
    if (k > 0) EG_TRY(lm_head_gemm(c, sink, c->hb, lo(c, c->hb_lo), c->ssq_b, M, k, nullptr));
    return EAGLE_OK;
  }

  static const ProgSpec* find_prog(eagle_ctx* c, int kind, int M, int hbase, int k) {
    for (const ProgSpec& p : c->dm.progs)
      if (p.kind == kind && p.M == M && p.hbase == hbase && p.k == k) return &p;
    return nullptr;
  }

  // Runs a recorded program; a program ending in the LM head merges its top-k
  // records in the same launch into idx / val / lse (k per row, as lm_head_merge).
  static eagle_status run_prog(eagle_ctx* c, const ProgSpec& p, float* lm_logits, int k, int* idx, float* val,
                               float* lse) {
    unsigned long long* trace = p.kind == 0 ? c->trace : nullptr;
    const Group* g = p.kind == 0 ? c->groups_local + p.seq0 : c->groups;
    const int ng = p.kind == 0 ? p.n_seq : c->dm.B;
    TopkMerge mg;
    if (k > 0) {
      mg.val = c->rec_val; mg.idx = c->rec_idx; mg.mx = c->rec_max; mg.sum = c->rec_sum;
      mg.ntiles = c->dm.ntV; mg.M = p.M; mg.k = k;
      mg.out_idx = idx; mg.out_val = val; mg.out_lse = lse;
    }
    EG_CK(stack_run(c->stack_prog + p.first, p.n_phases, p.M, pairs(c), c->dm.hd, p.n_counters,
                    c->stack_scratch, c->dm.stack_phases_max, c->dm.stack_counters_max, c->st.status, trace,
                    lm_logits, g, ng, p.first_attn, c->stream, p.w4, &mg));
    return EAGLE_OK;
  }

  // Record every program of the context into the workspace (at init).
  static eagle_status build_programs(eagle_ctx* c) {
    const Dims& dm = c->dm;
    if (sizeof(T) != 2 || dm.progs.empty()) return EAGLE_OK;
    std::vector<StackPhase> all;
    for (ProgSpec& p : c->dm.progs) {
      StackProgramBuilder b;
      b.M = p.M;
      b.MT = stack_mt(p.M);
      b.has_lo = pairs(c);
      Record r{c, &b};
      if (p.kind == 0) {
        EG_TRY(target_layers(c, r, p.M, p.n_seq, p.row0, c->groups_local + p.seq0));
        EG_TRY(lm_head_gemm(c, r, c->hb, lo(c, c->hb_lo), c->ssq_b, p.M, 1, nullptr, true, nullptr, p.row0));
      } else {
        EG_TRY(draft_ops(c, r, p.M, dm.B, p.hbase, p.k));
      }
      if ((int)b.phases.size() != p.n_phases || b.n_counters != p.n_counters)
        return fail(c, EAGLE_ERR_UNSUPPORTED, "persistent program: phase count");
      p.first_attn = b.first_attn;
      p.w4 = b.has_w4;
      all.insert(all.end(), b.phases.begin(), b.phases.end());
    }
    EG_CK(cudaMemcpyAsync(c->stack_prog, all.data(), all.size() * sizeof(StackPhase), cudaMemcpyHostToDevice,
                          c->stream));
    EG_CK(cudaStreamSynchronize(c->stream));  // `all` is a host temporary
    return EAGLE_OK;
  }

  // Fused-feature variant: fused[m] = fuse [low[m] ; mid[m] ; top[m]] for M rows (one GEMM, K = 3d).
  static eagle_status fuse_features(eagle_ctx* c, const float* low, const float* mid, const float* top, int M) {
    const Dims& dm = c->dm;
    EG_CK(pack_taps<T>(low, mid, top, M, dm.d, (T*)c->xfc, lo(c, c->xfc_lo), c->stream));
    EpiParams e = epi(c, kEpiStore, M, dm.d);
    e.y = c->fused;
    return gemm(c, c->xfc, lo(c, c->xfc_lo), c->fuse, M, dm.d, 3 * dm.d, e);
  }

  // Draft head over the phase's rows: FC([feature ; E(token)]) then the head layer, then (k > 0) LM-head top-k.
  static eagle_status draft_forward(eagle_ctx* c, const float* feat, int M, int n_groups, int hbase, int k) {
    const Dims& dm = c->dm;
    EG_CK(fc_input<T>(feat, c->rows.fsrc, (const T*)c->embed, c->rows.tok, M, dm.d, (T*)c->xfc, lo(c, c->xfc_lo),
                      c->stream));
    const ProgSpec* p = n_groups == dm.B ? find_prog(c, 1, M, hbase, k) : nullptr;
    if (p) {
      EG_TRY(run_prog(c, *p, nullptr, 0, nullptr, nullptr, nullptr));
    } else {
      Direct d{c};
      EG_TRY(draft_ops(c, d, M, n_groups, hbase, k));
    }
    // (the draft's top-10 merge stays a kernel of its own: merged inside the
    // persistent launch by one CTA per row, the 10 rows' merges made every draft
    // program tens of microseconds longer than the 512-thread merge kernel)
    if (k > 0)
      EG_TRY(lm_head_merge(c, M, k, c->dtopk_idx + (size_t)hbase * k, c->dtopk_val + (size_t)hbase * k,
                           c->dlse + hbase));
    return EAGLE_OK;
  }

  static eagle_status prefill(eagle_ctx* c, const int* d_tokens, int P, int* root_out) {
    const Dims& dm = c->dm;
    for (int c0 = 0; c0 < P; c0 += dm.CL) {
      const int cl = std::min(dm.CL, P - c0);
      const int M = dm.B * cl, G = dm.B * ((cl + 127) / 128);
      EG_CK(setup_prefill_rows(d_tokens, P, c0, cl, dm.B, false, c->rows, c->groups, c->stream));
      EG_TRY(target_stack(c, M, G));
      if (c0 + cl == P) {
        std::vector<int> src(dm.B);
        for (int b = 0; b < dm.B; ++b) src[b] = b * cl + cl - 1;
        EG_CK(cudaMemcpyAsync(c->lm_src, src.data(), dm.B * sizeof(int), cudaMemcpyHostToDevice, c->stream));
        EG_CK(gather_rows<T>((const T*)c->hb, lo(c, c->hb_lo), c->ssq_b, M, c->lm_src, dm.B, dm.d, (T*)c->lm_hb,
                             lo(c, c->lm_hb_lo), c->lm_ssq, c->stream));
        EG_TRY(lm_head(c, c->lm_hb, lo(c, c->lm_hb_lo), c->lm_ssq, dm.B, 1, c->root_idx, nullptr, nullptr, nullptr,
                       true, c->lm_src));
        EG_CK(prefill_finish(c->st, c->root_idx, c->h_tgt, c->h_low, c->h_mid, cl, P, root_out, c->stream));
        EG_CK(cudaStreamSynchronize(c->stream));  // src is a host temporary
      }
      EG_CK(setup_prefill_rows(d_tokens, P, c0, cl, dm.B, true, c->rows, c->groups, c->stream));
      if (dm.taps) EG_TRY(fuse_features(c, c->h_low, c->h_mid, c->h_tgt, M));
      EG_TRY(draft_forward(c, dm.taps ? c->fused : c->h_tgt, M, G, 0, 0));
    }
    return EAGLE_OK;
  }

  static eagle_status draft(eagle_ctx* c) {
    const Dims& dm = c->dm;
    const Level catchup{0, dm.D1};
    EG_CK(setup_catchup_rows(c->st, c->rows, c->groups, c->stream));
    if (dm.taps) EG_TRY(fuse_features(c, c->st.pend_low, c->st.pend_mid, c->st.pend_feat, dm.B * dm.D1));
    EG_TRY(draft_forward(c, dm.taps ? c->fused : c->st.pend_feat, dm.B * dm.D1, dm.B, 0, dm.k));
    for (int t = 1; t <= dm.D; ++t) {
      const Level prev = t > 1 ? Level{dm.level_base[t - 1], dm.level_rows[t - 1]} : Level{0, 0};
      const Level next = t < dm.D ? Level{dm.level_base[t], dm.level_rows[t]} : Level{0, 0};
      if (dm.mode == EAGLE_TREE_STATIC) {
        EG_CK(static_level(c->st, c->topo, t, c->dtopk_idx, c->dtopk_val, c->dlse, catchup, prev, next, c->tree,
                           c->rows, c->groups, dm.S, c->stream));
      } else {
        const float ln_tau = (float)std::log((double)c->cfg.tau);
        EG_CK(eagle2_level(c->st, c->pool, t, dm.D, dm.k, ln_tau, c->dtopk_idx, c->dtopk_val, c->dlse, catchup,
                           prev, next, c->rows, c->groups, dm.S, c->stream));
      }
      if (next.per_seq > 0)
        EG_TRY(draft_forward(c, c->h_dft, dm.B * next.per_seq, dm.B, next.base, dm.k));
    }
    if (dm.mode == EAGLE_TREE_DYNAMIC)
      EG_CK(eagle2_final(c->st, c->pool, dm.n_nodes, c->cfg.n_nodes_min, (float)std::log((double)c->cfg.tau), c->tree,
                         c->stream));
    return EAGLE_OK;
  }

  static eagle_status verify(eagle_ctx* c, const TreeOut& tree, int* d_argmax, float* d_logits) {
    const Dims& dm = c->dm;
    const int M = dm.B * tree.n_rows;
    EG_CK(setup_verify_rows(c->st, tree, c->rows, c->groups, c->groups_local, dm.verify_spc, c->stream));
    bool persistent = false;
    if (tree.n_rows == dm.NR)
      for (const ProgSpec& p : dm.progs)
        if (p.kind == 0) {
          // one persistent launch for every layer and the LM head (which also stores the logits if
          // wanted), per chunk of the batch when its rows exceed one launch
          EG_TRY(embed(c, p.M, p.row0));
          EG_TRY(run_prog(c, p, d_logits ? d_logits + (size_t)p.row0 * dm.V : nullptr, 1, c->vargmax + p.row0,
                          nullptr, nullptr));  // merge included
          persistent = true;
        }
    if (!persistent) {
      EG_TRY(target_stack(c, M, dm.B));
      EG_TRY(lm_head(c, c->hb, lo(c, c->hb_lo), c->ssq_b, M, 1, c->vargmax, nullptr, nullptr, d_logits, true));
    }
    if (d_argmax)
      EG_CK(cudaMemcpyAsync(d_argmax, c->vargmax, (size_t)M * sizeof(int), cudaMemcpyDeviceToDevice, c->stream));
    return EAGLE_OK;
  }

  static eagle_status accept(eagle_ctx* c, int* acc_out, int* tok_out) {
    const Dims& dm = c->dm;
    EG_CK(accept_commit(c->st, c->last_tree, c->vargmax, c->h_tgt, c->h_low, c->h_mid, acc_out, tok_out, c->stream));
    using KvT = typename KvOf<T>::type;
    EG_CK(compact_kv<KvT>(c->st, (KvT*)c->kc, (KvT*)c->vc, dm.Lyr, dm.Hkv, dm.hd, c->stream));
    return EAGLE_OK;
  }
};

template <typename F>
eagle_status dispatch(eagle_ctx* c, F&& f) {
  if (c->dm.bf16) return f(Eng<bf16>{});
  return f(Eng<float>{});
}

eagle_status check_ready(eagle_ctx* c) {
  if (!c) return EAGLE_ERR_INVALID_ARG;
  if (c->failed) return EAGLE_ERR_STATE;
  return EAGLE_OK;
}

eagle_status read_status(eagle_ctx* c) {
  int s = 0;
  EG_CK(cudaStreamSynchronize(c->stream));
  EG_CK(cudaMemcpy(&s, c->st.status, sizeof(int), cudaMemcpyDeviceToHost));
  if (s == kStCapacity) return fail(c, EAGLE_ERR_CAPACITY, "device: KV cache capacity exceeded");
  if (s == kStInvalid) {
    // the status word stays set and nothing was committed: the context is spent
    fail(c, EAGLE_ERR_INVALID_ARG, "device: verified tree is inconsistent or has two siblings with one token, "
                                   "or its accepted path is longer than the configured depth");
    c->failed = true;
    return EAGLE_ERR_INVALID_ARG;
  }
  if (s == kStTimeout) return fail(c, EAGLE_ERR_TIMEOUT, "device: bounded wait timed out");
  if (s != 0) return fail(c, EAGLE_ERR_CUDA, "device: status " + std::to_string(s));
  return EAGLE_OK;
}

}  // namespace
}  // namespace eg

using namespace eg;

extern "C" {

eagle_status eagle_workspace_size(const eagle_config* cfg, size_t* bytes) {
  if (!cfg || !bytes) return EAGLE_ERR_INVALID_ARG;
  Dims dm;
  std::string why;
  eagle_status s = derive(*cfg, dm, why);
  if (s != EAGLE_OK) return s;
  *bytes = plan(dm).total;
  return EAGLE_OK;
}

eagle_status eagle_init(const eagle_config* cfg, const eagle_weights* w, void* d_ws, size_t ws_bytes, void* stream,
                        eagle_ctx** out) {
  if (!cfg || !w || !out) return EAGLE_ERR_INVALID_ARG;
  *out = nullptr;
  eagle_ctx* c = new eagle_ctx();
  c->cfg = *cfg;
  std::string why;
  eagle_status s = derive(*cfg, c->dm, why);
  if (s != EAGLE_OK) {
    delete c;
    return s;
  }
  const Dims& dm = c->dm;
  if (!w->embed || !w->lm_head || !w->final_norm || !w->layers || !w->fc || (dm.taps && !w->fuse)) {
    delete c;
    return EAGLE_ERR_INVALID_ARG;
  }
  auto lp = [](const eagle_layer_weights& l, bool w4) {
    return LayerPtrs{l.wqkv, l.wo, l.wgu, l.wd, l.attn_norm, l.ffn_norm, w4};
  };
  for (int l = 0; l < dm.Lyr; ++l) c->layers.push_back(lp(w->layers[l], dm.w4));
  c->head = lp(w->head, false);
  if (dm.w4)
    for (const LayerPtrs& l : c->layers)
      if ((reinterpret_cast<uintptr_t>(l.wqkv) | reinterpret_cast<uintptr_t>(l.wo) |
           reinterpret_cast<uintptr_t>(l.wgu) | reinterpret_cast<uintptr_t>(l.wd)) & 15) {
        delete c;
        return EAGLE_ERR_INVALID_ARG;
      }
  for (const LayerPtrs& l : c->layers)
    if (!l.wqkv || !l.wo || !l.wgu || !l.wd || !l.attn_norm || !l.ffn_norm) { delete c; return EAGLE_ERR_INVALID_ARG; }
  if (!c->head.wqkv || !c->head.wo || !c->head.wgu || !c->head.wd || !c->head.attn_norm || !c->head.ffn_norm) {
    delete c;
    return EAGLE_ERR_INVALID_ARG;
  }
  c->embed = w->embed; c->lm_head = w->lm_head; c->final_norm = w->final_norm; c->fc = w->fc;
  c->fuse = dm.taps ? w->fuse : nullptr;
  const Offsets o = plan(dm);
  if (!d_ws || ws_bytes < o.total || (reinterpret_cast<uintptr_t>(d_ws) % kAlign)) {
    delete c;
    return EAGLE_ERR_WORKSPACE;
  }
  c->stream = (cudaStream_t)stream;
  char* base = (char*)d_ws;
  auto P = [&](size_t off) { return (void*)(base + off); };
  c->rows = Rows{(int*)P(o.rows_seq), (int*)P(o.rows_pos), (int*)P(o.rows_slot), (int*)P(o.rows_grp),
                 (uint64_t*)P(o.rows_mask), (int*)P(o.rows_tok), (int*)P(o.rows_fsrc)};
  c->groups = (Group*)P(o.groups);
  c->groups_local = (Group*)P(o.groups_local);
  c->h_tgt = (float*)P(o.h_tgt); c->h_dft = (float*)P(o.h_dft); c->hb = P(o.hb);
  if (dm.taps) {
    c->h_low = (float*)P(o.h_low); c->h_mid = (float*)P(o.h_mid); c->fused = (float*)P(o.fused);
  }
  c->ssq_a = (float*)P(o.ssq_a); c->ssq_b = (float*)P(o.ssq_b);
  c->q = P(o.q); c->qg = (__half*)P(o.qg); c->attn = P(o.attn); c->act = P(o.act); c->xfc = P(o.xfc);
  c->lm_hb = P(o.lm_hb); c->lm_ssq = (float*)P(o.lm_ssq); c->lm_src = (int*)P(o.lm_src);
  c->hb_lo = (bf16*)P(o.hb_lo); c->act_lo = (bf16*)P(o.act_lo); c->attn_lo = (bf16*)P(o.attn_lo);
  c->xfc_lo = (bf16*)P(o.xfc_lo); c->lm_hb_lo = (bf16*)P(o.lm_hb_lo);
  c->rec_val = (float*)P(o.rec_val); c->rec_idx = (int*)P(o.rec_idx);
  c->rec_max = (float*)P(o.rec_max); c->rec_sum = (float*)P(o.rec_sum);
  c->dtopk_idx = (int*)P(o.dtopk_idx); c->dtopk_val = (float*)P(o.dtopk_val); c->dlse = (float*)P(o.dlse);
  c->vargmax = (int*)P(o.vargmax); c->root_idx = (int*)P(o.root_idx);
  c->tree = TreeOut{dm.NR, (int*)P(o.t_tok), (int*)P(o.t_par), (int*)P(o.t_dep), (uint64_t*)P(o.t_anc),
                    (float*)P(o.t_score)};
  c->vtree = TreeOut{1, (int*)P(o.vt_tok), (int*)P(o.vt_par), (int*)P(o.vt_dep), (uint64_t*)P(o.vt_anc), nullptr};
  State& st = c->st;
  st.L = (int*)P(o.L); st.c = (int*)P(o.c); st.root = (int*)P(o.root); st.pend_tok = (int*)P(o.pend_tok);
  st.pend_feat = (float*)P(o.pend_feat);
  st.pend_low = dm.taps ? (float*)P(o.pend_low) : nullptr;
  st.pend_mid = dm.taps ? (float*)P(o.pend_mid) : nullptr; st.n_out = (int*)P(o.n_out); st.out = (int*)P(o.out);
  st.acc_len = (int*)P(o.acc_len); st.acc_path = (int*)P(o.acc_path); st.L_prev = (int*)P(o.L_prev);
  st.hist = (unsigned long long*)P(o.hist); st.status = (int*)P(o.status);
  st.B = dm.B; st.D1 = dm.D1; st.d = dm.d; st.cap = dm.cap; st.cap_d = dm.cap_d; st.out_cap = dm.out_cap;
  st.V = dm.V;
  Pool& pl = c->pool;
  pl.score = (float*)P(o.p_score); pl.token = (int*)P(o.p_token); pl.parent = (int*)P(o.p_parent);
  pl.depth = (int*)P(o.p_depth); pl.cid = (int*)P(o.p_cid); pl.frow = (int*)P(o.p_frow);
  pl.smask = (uint64_t*)P(o.p_smask); pl.count = (int*)P(o.p_count); pl.front = (int*)P(o.p_front);
  pl.nfront = (int*)P(o.p_nfront); pl.cap = dm.pool_cap;
  StaticTopo& tp = c->topo;
  tp.n_rows = dm.NR; tp.depth_max = dm.D; tp.k = dm.k;
  tp.parent = (int*)P(o.s_parent); tp.rank = (int*)P(o.s_rank); tp.depth = (int*)P(o.s_depth);
  tp.lrow = (int*)P(o.s_lrow); tp.sidx = (int*)P(o.s_sidx); tp.smask = (uint64_t*)P(o.s_smask);
  tp.level_nodes = (int*)P(o.s_lnodes); tp.level_count = (int*)P(o.s_lcount);
  c->rope_cos = (float*)P(o.rope_cos); c->rope_sin = (float*)P(o.rope_sin);
  c->kc = P(o.kc); c->vc = P(o.vc); c->kc_d = P(o.kc_d); c->vc_d = P(o.vc_d);
  c->gemm_scratch = P(o.gemm); c->gemm_scratch_bytes = o.gemm_bytes; c->attn_part = (float*)P(o.attn_part);
  c->stack_prog = (StackPhase*)P(o.stack_prog); c->stack_scratch = P(o.stack_scratch);
  c->stack_part = (float*)P(o.stack_part);
  c->w4_dense = dm.w4 ? P(o.w4_dense) : nullptr;

  // Zero the workspace (tile counters, status, caches), then upload the tables.
  cudaError_t e = cudaMemsetAsync(d_ws, 0, o.total, c->stream);
  // RoPE table: angle pos * theta^(-2i/hd), in double, rounded to float.
  const int half = dm.hd / 2;
  std::vector<float> cs((size_t)dm.cap_d * half), sn((size_t)dm.cap_d * half);
  for (int p = 0; p < dm.cap_d; ++p)
    for (int i = 0; i < half; ++i) {
      const double inv = std::pow((double)cfg->rope_theta, -2.0 * i / dm.hd);
      const double ang = (double)p * inv;
      cs[(size_t)p * half + i] = (float)std::cos(ang);
      sn[(size_t)p * half + i] = (float)std::sin(ang);
    }
  if (e == cudaSuccess) e = cudaMemcpyAsync(c->rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice, c->stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(c->rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice, c->stream);
  std::vector<int> tpar, tdep;
  std::vector<uint64_t> tanc;
  if (e == cudaSuccess && dm.mode == EAGLE_TREE_STATIC) {
    const size_t NR = dm.NR;
    e = cudaMemcpyAsync((void*)tp.parent, dm.s_parent.data(), NR * 4, cudaMemcpyHostToDevice, c->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync((void*)tp.rank, dm.s_rank.data(), NR * 4, cudaMemcpyHostToDevice, c->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync((void*)tp.depth, dm.s_depth.data(), NR * 4, cudaMemcpyHostToDevice, c->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync((void*)tp.lrow, dm.s_lrow.data(), NR * 4, cudaMemcpyHostToDevice, c->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync((void*)tp.sidx, dm.s_sidx.data(), NR * 4, cudaMemcpyHostToDevice, c->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync((void*)tp.smask, dm.s_smask.data(), NR * 8, cudaMemcpyHostToDevice, c->stream);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync((void*)tp.level_nodes, dm.s_level_nodes.data(), dm.s_level_nodes.size() * 4,
                          cudaMemcpyHostToDevice, c->stream);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync((void*)tp.level_count, dm.s_level_count.data(), dm.s_level_count.size() * 4,
                          cudaMemcpyHostToDevice, c->stream);
    for (int b = 0; b < dm.B; ++b) {
      tpar.insert(tpar.end(), dm.s_parent.begin(), dm.s_parent.end());
      tdep.insert(tdep.end(), dm.s_depth.begin(), dm.s_depth.end());
      tanc.insert(tanc.end(), dm.s_anc.begin(), dm.s_anc.end());
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(c->tree.parent, tpar.data(), tpar.size() * 4, cudaMemcpyHostToDevice, c->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(c->tree.depth, tdep.data(), tdep.size() * 4, cudaMemcpyHostToDevice, c->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(c->tree.anc, tanc.data(), tanc.size() * 8, cudaMemcpyHostToDevice, c->stream);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
  if (e != cudaSuccess) {
    delete c;
    return EAGLE_ERR_CUDA;
  }
  const eagle_status ps = dispatch(c, [&](auto E) { return decltype(E)::build_programs(c); });
  if (ps != EAGLE_OK) {
    delete c;
    return ps;
  }
  *out = c;
  return EAGLE_OK;
}

eagle_status eagle_prefill(eagle_ctx* c, const int32_t* d_tokens, int32_t P, int32_t* d_root_out) {
  EG_TRY(check_ready(c));
  if (!d_tokens || P < 1 || P > c->dm.P_max) return fail(c, EAGLE_ERR_INVALID_ARG, "prompt_len out of range");
  EG_TRY(dispatch(c, [&](auto E) { return decltype(E)::prefill(c, d_tokens, P, d_root_out); }));
  c->phase = 1;
  return EAGLE_OK;
}

eagle_status eagle_draft_tree(eagle_ctx* c, eagle_tree* out) {
  EG_TRY(check_ready(c));
  if (c->phase < 1) return fail(c, EAGLE_ERR_INVALID_ARG, "draft before prefill");
  if (c->phase == 2 || c->phase == 3) return fail(c, EAGLE_ERR_INVALID_ARG, "draft twice without accept");
  EG_TRY(dispatch(c, [&](auto E) { return decltype(E)::draft(c); }));
  if (out && out->tokens) {
    if (!out->parent || !out->depth || !out->anc || out->n_rows < c->tree.n_rows)
      return fail(c, EAGLE_ERR_INVALID_ARG, "draft_tree: caller arrays too small");
    const size_t n = (size_t)c->dm.B * c->tree.n_rows;
    // caller arrays use the same [batch][n_rows] packing as the workspace tree
    EG_CK(cudaMemcpyAsync(out->tokens, c->tree.tokens, n * 4, cudaMemcpyDeviceToDevice, c->stream));
    EG_CK(cudaMemcpyAsync(out->parent, c->tree.parent, n * 4, cudaMemcpyDeviceToDevice, c->stream));
    EG_CK(cudaMemcpyAsync(out->depth, c->tree.depth, n * 4, cudaMemcpyDeviceToDevice, c->stream));
    EG_CK(cudaMemcpyAsync(out->anc, c->tree.anc, n * 16, cudaMemcpyDeviceToDevice, c->stream));
    if (out->score) EG_CK(cudaMemcpyAsync(out->score, c->tree.score, n * 4, cudaMemcpyDeviceToDevice, c->stream));
    out->n_rows = c->tree.n_rows;
  } else if (out) {
    *out = eagle_tree{c->tree.n_rows, c->tree.tokens, c->tree.parent, c->tree.depth, c->tree.anc, c->tree.score};
  }
  c->phase = 2;
  return EAGLE_OK;
}

eagle_status eagle_verify(eagle_ctx* c, const eagle_tree* tree, int32_t* d_argmax, float* d_logits) {
  EG_TRY(check_ready(c));
  if (c->phase < 1) return fail(c, EAGLE_ERR_INVALID_ARG, "verify before prefill");
  if (!tree || tree->n_rows < 1 || tree->n_rows > EAGLE_MAX_TREE_ROWS || !tree->tokens || !tree->parent ||
      !tree->depth || !tree->anc)
    return fail(c, EAGLE_ERR_INVALID_ARG, "bad tree");
  TreeOut t{tree->n_rows, tree->tokens, tree->parent, tree->depth, tree->anc, nullptr};
  c->last_tree = t;
  EG_TRY(dispatch(c, [&](auto E) { return decltype(E)::verify(c, t, d_argmax, d_logits); }));
  c->phase = 3;
  return EAGLE_OK;
}

eagle_status eagle_accept_commit(eagle_ctx* c, int32_t* d_accept_len, int32_t* d_tokens_out) {
  EG_TRY(check_ready(c));
  if (c->phase != 3) return fail(c, EAGLE_ERR_INVALID_ARG, "accept without verify");
  EG_TRY(dispatch(c, [&](auto E) { return decltype(E)::accept(c, d_accept_len, d_tokens_out); }));
  c->phase = 1;
  return EAGLE_OK;
}

static eagle_status step_once(eagle_ctx* c, bool vanilla) {
  return dispatch(c, [&](auto E) -> eagle_status {
    using En = decltype(E);
    if (vanilla) {
      const TreeOut t = c->vtree;
      EG_CK(set_root_tree(c->st, t, c->stream));
      c->last_tree = t;
      EG_TRY(En::verify(c, t, nullptr, nullptr));
    } else {
      EG_TRY(En::draft(c));
      c->last_tree = c->tree;
      EG_TRY(En::verify(c, c->tree, nullptr, nullptr));
    }
    return En::accept(c, nullptr, nullptr);
  });
}

// The captured step of this context (captured on first use). A legacy-default
// (NULL) stream cannot be captured: *exec stays NULL and the caller runs eagerly.
static eagle_status step_graph(eagle_ctx* c, bool vanilla, cudaGraphExec_t* exec) {
  *exec = nullptr;
  if (c->stream == nullptr) return EAGLE_OK;
  cudaGraphExec_t& slot = c->graph_exec[vanilla ? 1 : 0];
  if (!slot) {
    cudaGraph_t graph = nullptr;
    EG_CK(cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal));
    eagle_status s = step_once(c, vanilla);
    cudaError_t ce = cudaStreamEndCapture(c->stream, &graph);
    if (s != EAGLE_OK) {
      if (graph) cudaGraphDestroy(graph);
      return s;
    }
    if (ce != cudaSuccess) return fail(c, EAGLE_ERR_CUDA, std::string("graph capture: ") + cudaGetErrorString(ce));
    size_t n_nodes = 0;
    EG_CK(cudaGraphGetNodes(graph, nullptr, &n_nodes));
    std::vector<cudaGraphNode_t> nodes(n_nodes);
    EG_CK(cudaGraphGetNodes(graph, nodes.data(), &n_nodes));
    int kernels = 0;
    for (cudaGraphNode_t nd : nodes) {
      cudaGraphNodeType ty;
      EG_CK(cudaGraphNodeGetType(nd, &ty));
      kernels += ty == cudaGraphNodeTypeKernel;
    }
    c->graph_kernels[vanilla ? 1 : 0] = kernels;
    cudaError_t ie = cudaGraphInstantiate(&slot, graph, 0);
    cudaGraphDestroy(graph);
    if (ie != cudaSuccess) return fail(c, EAGLE_ERR_CUDA, std::string("graph instantiate: ") + cudaGetErrorString(ie));
  }
  *exec = slot;
  return EAGLE_OK;
}

static eagle_status run_steps(eagle_ctx* c, int n, bool vanilla, cudaGraphExec_t exec) {
  for (int i = 0; i < n; ++i) {
    if (exec) {
      EG_CK(cudaGraphLaunch(exec, c->stream));
    } else {
      EG_TRY(step_once(c, vanilla));
    }
  }
  return EAGLE_OK;
}

static eagle_status generate(eagle_ctx* c, const int32_t* d_prompt, int32_t P, int32_t max_new, int32_t use_graph,
                             int32_t* d_out, eagle_stats* h_stats, bool vanilla) {
  EG_TRY(check_ready(c));
  const Dims& dm = c->dm;
  if (!d_prompt || !d_out || P < 1 || P > dm.P_max || max_new < 1 || max_new > c->cfg.max_new)
    return fail(c, EAGLE_ERR_INVALID_ARG, "generate: bad arguments");
  cudaEvent_t e0, e1, e2;
  EG_CK(cudaEventCreate(&e0));
  EG_CK(cudaEventCreate(&e1));
  EG_CK(cudaEventCreate(&e2));
  EG_CK(cudaMemsetAsync(c->st.hist, 0, (kMaxDepth + 1) * 8, c->stream));
  EG_CK(cudaEventRecord(e0, c->stream));
  EG_TRY(dispatch(c, [&](auto E) { return decltype(E)::prefill(c, d_prompt, P, nullptr); }));
  c->phase = 1;
  EG_CK(cudaEventRecord(e1, c->stream));
  cudaGraphExec_t exec = nullptr;
  if (use_graph) EG_TRY(step_graph(c, vanilla, &exec));
  std::vector<int> nout(dm.B);
  int64_t steps = 0;
  double tps = 1.0;
  for (;;) {
    EG_CK(cudaMemcpyAsync(nout.data(), c->st.n_out, dm.B * sizeof(int), cudaMemcpyDeviceToHost, c->stream));
    EG_CK(cudaStreamSynchronize(c->stream));
    int mn = nout[0];
    long long tot = 0;
    for (int b = 0; b < dm.B; ++b) { mn = std::min(mn, nout[b]); tot += nout[b]; }
    if (mn >= max_new) break;
    if (steps > 0) tps = std::max(1.0, (double)(tot - dm.B) / (double)(steps * dm.B));
    const int remaining = max_new - mn;
    int run = std::max(1, (int)std::floor(remaining / tps));
    if (steps == 0) run = std::min(run, 8);
    EG_TRY(run_steps(c, run, vanilla, exec));
    steps += run;
    if (steps > (int64_t)max_new * 2 + 16) return fail(c, EAGLE_ERR_STATE, "generate: no progress");
  }
  EG_CK(cudaEventRecord(e2, c->stream));
  EG_CK(copy_out(c->st, max_new, d_out, c->stream));
  eagle_status s = read_status(c);
  if (s != EAGLE_OK) return s;
  if (h_stats) {
    std::memset(h_stats, 0, sizeof(*h_stats));
    unsigned long long hist[kMaxDepth + 1];
    EG_CK(cudaMemcpy(hist, c->st.hist, sizeof(hist), cudaMemcpyDeviceToHost));
    int64_t n = 0, acc = 0;
    for (int i = 0; i <= kMaxDepth; ++i) {
      h_stats->accept_hist[i] = (int64_t)hist[i];
      n += (int64_t)hist[i];
      acc += (int64_t)hist[i] * i;
    }
    h_stats->steps = steps;
    h_stats->mean_accept = n ? (double)acc / n : 0.0;
    EG_CK(cudaMemcpy(nout.data(), c->st.n_out, dm.B * sizeof(int), cudaMemcpyDeviceToHost));
    for (int b = 0; b < dm.B; ++b) h_stats->committed += nout[b];
    float ms = 0.f;
    EG_CK(cudaEventElapsedTime(&ms, e0, e1));
    h_stats->prefill_ms = ms;
    EG_CK(cudaEventElapsedTime(&ms, e1, e2));
    h_stats->decode_ms = ms;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaEventDestroy(e2);
  return EAGLE_OK;
}

eagle_status eagle_generate(eagle_ctx* c, const int32_t* d_prompt, int32_t P, int32_t max_new, int32_t use_graph,
                            int32_t* d_out, eagle_stats* h_stats) {
  return generate(c, d_prompt, P, max_new, use_graph, d_out, h_stats, false);
}

eagle_status eagle_generate_vanilla(eagle_ctx* c, const int32_t* d_prompt, int32_t P, int32_t max_new,
                                    int32_t use_graph, int32_t* d_out, eagle_stats* h_stats) {
  return generate(c, d_prompt, P, max_new, use_graph, d_out, h_stats, true);
}

eagle_status eagle_step(eagle_ctx* c, int32_t n_steps, int32_t vanilla, int32_t use_graph) {
  EG_TRY(check_ready(c));
  if (c->phase != 1) return fail(c, EAGLE_ERR_INVALID_ARG, "step: needs a prefilled context between steps");
  if (n_steps < 0) return fail(c, EAGLE_ERR_INVALID_ARG, "step: n_steps < 0");
  cudaGraphExec_t exec = nullptr;
  if (use_graph) EG_TRY(step_graph(c, vanilla != 0, &exec));
  return run_steps(c, n_steps, vanilla != 0, exec);
}

int32_t eagle_step_kernel_count(const eagle_ctx* c, int32_t vanilla) {
  return c ? c->graph_kernels[vanilla ? 1 : 0] : -1;
}

eagle_status eagle_sync_status(eagle_ctx* c) {
  if (!c) return EAGLE_ERR_INVALID_ARG;
  if (c->failed) return EAGLE_ERR_STATE;
  return read_status(c);
}

eagle_status eagle_committed_counts(eagle_ctx* c, int32_t* d_counts) {
  if (!c || !d_counts) return EAGLE_ERR_INVALID_ARG;
  EG_CK(cudaMemcpyAsync(d_counts, c->st.n_out, c->dm.B * sizeof(int), cudaMemcpyDeviceToDevice, c->stream));
  return EAGLE_OK;
}

eagle_status eagle_set_trace(eagle_ctx* c, uint64_t* d_trace, size_t n, int32_t* n_phases, int32_t* n_ctas) {
  if (!c) return EAGLE_ERR_INVALID_ARG;
  const ProgSpec* v = nullptr;
  for (const ProgSpec& p : c->dm.progs)
    if (p.kind == 0) v = &p;
  const int ph = v ? v->n_phases : 0, ctas = v ? stack_ctas() : 0;
  if (n_phases) *n_phases = ph;
  if (n_ctas) *n_ctas = ctas;
  if (d_trace && (!v || n < (size_t)(ph + 1) * ctas)) return EAGLE_ERR_INVALID_ARG;
  c->trace = reinterpret_cast<unsigned long long*>(d_trace);
  // captured steps bake the trace pointer: drop them
  for (int i = 0; i < 2; ++i)
    if (c->graph_exec[i]) {
      cudaGraphExecDestroy(c->graph_exec[i]);
      c->graph_exec[i] = nullptr;
      c->graph_kernels[i] = -1;
    }
  return EAGLE_OK;
}

eagle_status eagle_destroy(eagle_ctx* c) {
  if (!c) return EAGLE_ERR_INVALID_ARG;
  for (cudaGraphExec_t& g : c->graph_exec)
    if (g) cudaGraphExecDestroy(g);
  delete c;
  return EAGLE_OK;
}

const char* eagle_last_error(const eagle_ctx* c) { return c ? c->err.c_str() : "null context"; }

size_t eagle_struct_size(int32_t which) {
  switch (which) {
    case 0: return sizeof(eagle_config);
    case 1: return sizeof(eagle_weights);
    case 2: return sizeof(eagle_layer_weights);
    case 3: return sizeof(eagle_tree);
    case 4: return sizeof(eagle_stats);
    default: return 0;
  }
}

}  // extern "C"
