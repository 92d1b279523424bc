// Persistent layer-stack forward (bf16 models, up to 128 token rows).
//
// One cooperative launch runs a whole program of phases - the GEMMs of every
// decoder layer with their fused epilogues, tree attention and its merge, and
// the LM head - on one CTA per SM. Phase p may read only what phases < p wrote;
// the kernel orders them with grid-wide arrival counters. The weight boxes of
// every GEMM phase do not depend on earlier phases, so each CTA's weight
// producer streams them ahead across phase boundaries; only the activation
// boxes of phase p wait for phase p - 1 to finish.
#pragma once

#include <vector>

#include "kernels.h"
#include "topk.cuh"

namespace eg {

enum StackPhaseKind : int { kPhaseGemm = 0, kPhaseAttn = 1, kPhaseMerge = 2 };

struct StackPhase {   // 128-byte aligned (CUtensorMap)
  CUtensorMap tmW;    // GEMM weight [N][K], box [128][64]; attention: K cache rows, box [128][64]
  CUtensorMap tmX;    // GEMM activations [rows][K], box [MT][64]; attention: V cache rows
  CUtensorMap tmXlo;  // low halves of the activations (hi/lo pair); attention: grouped half queries
  int kind = kPhaseGemm;
  int N = 0, K = 0, n_tiles = 0, kbt = 0;
  long long T = 0;    // units (128-row tile, 64-wide k-block): n_tiles * kbt
  int cnt_off = 0;    // first split-K arrival counter of this phase
  const uint8_t* w4 = nullptr;  // GEMM: packed int4 weight (int4.cuh blocks) instead of tmW
  EpiParams ep;       // GEMM epilogue
  AttnArgs at;        // attention / merge
};

// One GEMM phase: Y = (X + X_lo) W^T over the program's M rows, then epilogue ep.
struct StackGemmDesc {
  const bf16* W;
  const bf16* X;
  const bf16* X_lo;   // may be NULL
  int rows_cap;       // rows of the X buffers (>= M)
  int N, K;
  EpiParams ep;
  bool w4 = false;    // W is a packed int4 weight (int4.cuh block layout), expanded in shared memory
};

// Host-side builder of a program (tensor maps are encoded here).
struct StackProgramBuilder {
  int M = 0, MT = 0;
  bool has_lo = false;
  std::vector<StackPhase> phases;
  int n_counters = 0;
  int first_attn = -1;  // index of the first attention phase
  bool has_w4 = false;  // some GEMM phase has an int4 weight: run with stack_run(..., w4 = true)
  bool ok = true;
  void gemm(const StackGemmDesc& g);
  void attention(const AttnArgs& a);  // adds the attention phase and its merge phase
};

// Largest M the persistent kernel takes.
constexpr int kStackMaxRows = 128;
bool stack_supported(int M, int hd);
// Token rows of one MMA tile for M rows (the activation box height).
int stack_mt(int M);
// CTAs of one launch (one per SM).
int stack_ctas();
// Bytes of device scratch shared by programs of at most M rows, max_phases
// phases and max_counters split-K counters: phase counters, split-K counters,
// partial sums (zero-initialised by the caller once).
size_t stack_scratch_bytes(int M, int max_phases, int max_counters);
// Attention partial buffer of the persistent kernel.
size_t stack_attention_part_bytes(int M, int Hq, int Hkv, int hd, int max_prefix);
// Runs the program (d_phases: device copy of builder.phases) on stack_ctas()
// CTAs. scratch holds stack_scratch_bytes(M', max_phases, max_counters) bytes
// for capacities that every program sharing it fits (the layout is derived from
// them alone). Scratch counters must be zero on entry; the kernel leaves them zero.
// trace (may be NULL): [n_phases + 1][stack_ctas()] %globaltimer stamps - row p
// = when each CTA finished phase p, the last row = when it started.
// y_last (may be NULL): replaces the output pointer y of the last phase's
// epilogue for this launch (the LM head's optional logits).
// groups / n_groups (<= 128): the groups every attention phase of the program
// reads (each CTA keeps a copy in shared memory); NULL / 0 without attention.
// first_attn: index of the program's first attention phase (-1 if none); every
// attention phase of a program has the same rows, heads and groups.
// w4: the program has int4 phases (the 352-thread variant with converter warps).
// merge (may be NULL; merge->k == 0: none): the last phase is an LM head whose
// top-k records are merged in the same launch (merge->M <= M rows, CTA c taking
// row c once every CTA has finished that phase) instead of by topk_merge.
cudaError_t stack_run(const StackPhase* d_phases, int n_phases, int M, bool has_lo, int hd, int n_counters,
                      void* scratch, int max_phases, int max_counters, int* status, unsigned long long* trace,
                      float* y_last, const Group* groups, int n_groups, int first_attn, cudaStream_t s,
                      bool w4 = false, const TopkMerge* merge = nullptr);

}  // namespace eg
