/*
 * eagle.h - C ABI of the GB300 EAGLE speculative-decoding step.
 *
 * One speculative-decoding step of a Llama-style target model on one GPU:
 *   draft  (feature-level head + static or EAGLE-2 dynamic tree),
 *   verify (one tree-masked target pass over the KV cache),
 *   accept (greedy longest accepted root-to-leaf path),
 *   commit (compact the accepted K/V and features in place).
 *
 * Method sources (web pages on EAGLE speculative decoding):
 *   [SDE]  "Speculative Decoding with EAGLE" (aiunderstanding.org), sections
 *          "Deep dive" and "Technical insight".
 *   [LPD]  "EAGLE (LLM decoding)" (jisaku.com/glossary/llm-parallel-decoding-eagle),
 *          sections "How EAGLE works", "EAGLE vs EAGLE-2", FAQ Q3.
 *   [YHL]  "yuhuili" (llmyourway.com/authors/yuhuili).
 *
 * Conventions for every entry point:
 *   - All functions are `extern "C"`, never throw, and return eagle_status.
 *   - "d_" pointers are device pointers, "h_" pointers host pointers.
 *   - Work is enqueued asynchronously on the stream given to eagle_init
 *     (a cudaStream_t passed as void*; NULL selects the legacy default stream).
 *     Only eagle_generate, eagle_sync_status and eagle_op_* timing helpers
 *     synchronise that stream.
 *   - The library never allocates device memory: the caller owns the weights,
 *     the workspace (size from eagle_workspace_size) and all outputs, and keeps
 *     them alive until eagle_destroy.
 *   - Argument errors are detected on the host and returned synchronously.
 *     Errors found on the device (KV capacity, bounded-wait timeout) are
 *     written to a status word in the workspace and returned by the next
 *     eagle_sync_status / eagle_generate. After any error the context refuses
 *     further work with EAGLE_ERR_STATE until destroyed; eagle_last_error
 *     gives a one-line description.
 *
 * Data types: EAGLE_DTYPE_F32 models keep weights, activations and the KV
 * cache in float32 (SIMT kernels). EAGLE_DTYPE_BF16 models keep weights in
 * bfloat16, the KV cache in IEEE half (11-bit significand at two bytes;
 * stores saturate at +-65504), the residual stream, features, queries and
 * softmax statistics in float32, and feed every GEMM with activations split
 * into hi/lo bfloat16 pairs (x = hi + lo, two tensor-core products accumulated
 * in float32), so GEMM inputs carry ~16 significant bits (tcgen05 tensor-core
 * GEMMs); models with int4 target projections (weight_bits = 4) feed their
 * GEMMs plain bfloat16 activations instead (W4A16). Attention products are
 * half x half with float32 accumulation (tcgen05 tensor-core attention).
 */
#ifndef EAGLE_H
#define EAGLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EAGLE_OK = 0,
  EAGLE_ERR_INVALID_ARG = 1,   /* bad pointer, size or shape (host-detected) */
  EAGLE_ERR_UNSUPPORTED = 2,   /* shape the kernels do not support */
  EAGLE_ERR_WORKSPACE = 3,     /* workspace too small or misaligned */
  EAGLE_ERR_CAPACITY = 4,      /* KV cache or output capacity exceeded (device-detected) */
  EAGLE_ERR_CUDA = 5,          /* a CUDA runtime or driver call failed */
  EAGLE_ERR_TIMEOUT = 6,       /* a bounded device wait gave up */
  EAGLE_ERR_STATE = 7          /* call out of order, or context already failed */
} eagle_status;

typedef enum { EAGLE_DTYPE_F32 = 0, EAGLE_DTYPE_BF16 = 1 } eagle_dtype;
typedef enum { EAGLE_TREE_STATIC = 0, EAGLE_TREE_DYNAMIC = 1 } eagle_tree_mode;

/* Largest verified tree: 120 draft nodes plus the root ([LPD] "EAGLE vs
 * EAGLE-2": EAGLE-2 adapts between 40 and 120 nodes). Ancestor sets are
 * 128-bit masks. */
#define EAGLE_MAX_TREE_ROWS 121
#define EAGLE_MAX_DEPTH 8
#define EAGLE_MAX_TOPK 16

/* Model and decoding configuration. */
typedef struct {
  int32_t n_layers;      /* target decoder layers */
  int32_t d;             /* hidden size; multiple of 128 */
  int32_t n_heads;       /* query heads */
  int32_t n_kv_heads;    /* KV heads (grouped-query attention); divides n_heads */
  int32_t head_dim;      /* 64 or 128 */
  int32_t ffn;           /* SwiGLU inner size */
  int32_t vocab;         /* vocabulary size */
  float rope_theta;      /* RoPE base */
  float rms_eps;         /* RMSNorm epsilon */
  int32_t dtype;         /* eagle_dtype */
  int32_t batch;         /* independent sequences decoded together */
  int32_t kv_cap;        /* KV slots per sequence (prompt + generated + tree) */
  int32_t max_prompt;    /* longest prompt eagle_prefill will see */
  int32_t max_new;       /* capacity of the per-sequence committed-token buffer */
  int32_t tree_mode;     /* eagle_tree_mode */
  int32_t n_nodes;       /* verified draft nodes per step, root excluded (<= 120) */
  /* EAGLE_TREE_STATIC: BFS-ordered topology, host arrays of n_nodes+1 entries,
   * copied at eagle_init. static_parent[0] = -1 (root); static_rank[j] = r
   * makes node j the r-th most likely draft token of its parent. */
  const int32_t* static_parent;
  const int32_t* static_rank;
  /* EAGLE_TREE_DYNAMIC ([LPD] "EAGLE vs EAGLE-2", FAQ Q3): expand the top_k
   * nodes per depth by cumulative draft confidence, children top_k per node,
   * depth levels, prune expansion below confidence tau. */
  int32_t top_k;
  int32_t depth;
  float tau;
  /* The target's choice of each next token ([SDE] "Technical insight": a
   * drafted token is accepted when it matches the target's argmax, or its
   * sample): temperature 0 = greedy argmax; temperature T > 0 = a sample of
   * softmax(logits / T), drawn by the Gumbel-max rule with noise
   *   g = -log(-log(u)),  u = ((z >> 40) + 0.5) 2^-24,
   *   z = mix64(mix64(mix64(seed + (b+1) G) + (p+1) G) + (v+1) G),
   * for sequence b, token position p, vocabulary entry v (mix64 = SplitMix64's
   * output function, G = 0x9E3779B97F4A7C15). The noise depends on the position
   * only, so speculative sampling commits exactly the tokens vanilla sampling
   * with the same seed commits. The draft tree is built by draft top-k either way. */
  float temperature;
  uint64_t seed;
  /* EAGLE_TREE_DYNAMIC, adaptive node count ([LPD] "EAGLE vs EAGLE-2": 40-120
   * verified nodes instead of a fixed 60): when > 0, each sequence verifies the
   * pool candidates whose cumulative confidence reaches tau, at least n_nodes_min
   * and at most n_nodes of them (its tree's remaining rows are padding rows with
   * token -1); 0 = every sequence verifies n_nodes. */
  int32_t n_nodes_min;
  /* The feature the draft head takes for committed positions ([LPD], the
   * EAGLE-3 entry: the draft fuses low-, mid- and high-level target features;
   * the page gives no layer choice, read here as): 0 or 1 = the target's top-layer
   * feature (EAGLE, EAGLE-2); 3 = u = fuse [f_low ; f_mid ; f_top], the hidden
   * states after target layers max(1, n_layers/4), max(1, n_layers/2) and
   * n_layers (eagle_weights.fuse is then required). The target's own logits
   * always come from its top-layer feature. */
  int32_t feature_taps;
  /* Weights of the target's decoder-layer projections ([LPD] operational notes:
   * EAGLE combines with GPTQ / AWQ 4-bit weight-quantised targets): 0 or 16 =
   * `dtype` elements; 4 = weight-only int4 (each of wqkv, wo, wgu, wd points to
   * eagle_int4_pack's block layout; symmetric, a bf16 scale per row and group of
   * 64 inputs, W = bf16(scale * (code - 8))). Activations are plain bf16 (no
   * hi/lo pairs: W4A16); the
   * embedding, LM head, norms and the draft head are not quantised. Needs d, the
   * query width and ffn to be multiples of 64. */
  int32_t weight_bits;
} eagle_config;

/* Device pointers of one decoder layer. Matrices are row-major [out, in]
 * (y = x W^T), element type = config dtype; norm gains are float32 [d]. */
typedef struct {
  const void* wqkv;        /* [(n_heads + 2 n_kv_heads) head_dim, d]: q rows, then k, then v */
  const void* wo;          /* [d, n_heads head_dim] */
  const void* wgu;         /* [2 ffn, d]: gate and up rows interleaved in blocks of 64:
                              block b holds gate rows 64b.. then up rows 64b.. (the last
                              block may hold r < 64 of each) */
  const void* wd;          /* [d, ffn] */
  const float* attn_norm;  /* [d] */
  const float* ffn_norm;   /* [d] */
} eagle_layer_weights;

typedef struct {
  const void* embed;                   /* [vocab, d] token embedding E */
  const void* lm_head;                 /* [vocab, d] */
  const float* final_norm;             /* [d] */
  const eagle_layer_weights* layers;   /* host array of n_layers entries */
  const void* fc;                      /* draft head FC [d, 2d] over [feature ; E(next token)] */
  eagle_layer_weights head;            /* draft head decoder layer */
  const void* fuse;                    /* feature_taps = 3: [d, 3d] over [f_low ; f_mid ; f_top]; else unused */
} eagle_weights;

/* A draft tree per sequence, BFS order, row 0 = root. Device arrays.
 * A tree passed to eagle_verify must be consistent: parent[0] = -1, depth[0] = 0,
 * anc[0] = {1, 0}; for j > 0, 0 <= parent[j] < j, depth[j] = depth[parent[j]] + 1,
 * anc[j] = anc[parent[j]] | bit j; and siblings carry distinct tokens (rows
 * with token -1 are padding, never accepted, and come after every real row),
 * so that the greedy accepted path is unique. Trees deeper than the configured tree depth may be verified (for
 * example a chain carrying a known continuation, to read its logits), but
 * eagle_accept_commit refuses an accepted path longer than that depth. */
typedef struct {
  int32_t n_rows;          /* N + 1, same for every sequence */
  int32_t* tokens;         /* [batch][n_rows] */
  int32_t* parent;         /* [batch][n_rows], -1 at the root */
  int32_t* depth;          /* [batch][n_rows] */
  uint64_t* anc;           /* [batch][n_rows][2]: bit i set when row i is on the root-to-row path (self included) */
  float* score;            /* [batch][n_rows] or NULL: cumulative draft log-confidence of each row, the sum of
                              the draft log-probabilities along its root-to-row path ([LPD] "EAGLE vs EAGLE-2";
                              0 at the root, -inf at padding rows); written by eagle_draft_tree, unused by
                              eagle_verify */
} eagle_tree;

typedef struct {
  int64_t steps;               /* speculative steps run by eagle_generate */
  int64_t committed;           /* tokens committed over all sequences (before trimming) */
  int64_t accept_hist[EAGLE_MAX_DEPTH + 1]; /* accepted draft length per (step, sequence) */
  double mean_accept;          /* mean accepted draft tokens per step and sequence */
  double prefill_ms;           /* wall time of the prefill */
  double decode_ms;            /* wall time of the step loop */
} eagle_stats;

typedef struct eagle_ctx eagle_ctx;

/* Bytes of device workspace eagle_init needs for this configuration. Host-only; no CUDA call. */
eagle_status eagle_workspace_size(const eagle_config* cfg, size_t* bytes);
/* (The workspace holds the KV caches of the target and the head, the rows of
 * every forward, the decoding state and the kernels' scratch; [SDE] "Deep
 * dive": the KV cache of the verified prefix is reused across steps.) */

/* Validate the configuration, carve the workspace (256-byte aligned, owned by
 * the caller, contents overwritten) and bind the weights: the target decoder
 * stack, and the draft head that shares its embedding, final norm and LM head
 * ([SDE] "Technical insight": the head reuses the target's own LM head; [LPD]
 * "How EAGLE works": a one-layer head over the target's top-layer feature).
 * Returns the context through *out. The device current at this call must be
 * the one holding all pointers. */
eagle_status eagle_init(const eagle_config* cfg, const eagle_weights* w, void* d_workspace,
                        size_t workspace_bytes, void* stream, eagle_ctx** out);

/* Target prefill of batch prompts of equal length prompt_len (d_tokens
 * [batch][prompt_len]; ragged prompts are not supported), the head's rows over
 * prompt positions 0..prompt_len-2 (feature f_i with the embedding of the next
 * true token t_{i+1}: [SDE] "Technical insight", the shifted token sequence),
 * and the first new token (greedy) per sequence, written to d_root_out [batch]
 * when not NULL. Resets all per-sequence state. */
eagle_status eagle_prefill(eagle_ctx* ctx, const int32_t* d_tokens, int32_t prompt_len,
                           int32_t* d_root_out);

/* Draft step ([SDE] "Technical insight"; [LPD] "How EAGLE works", "EAGLE vs
 * EAGLE-2"): head rows for the positions committed last, then tree expansion
 * (static rank paths or EAGLE-2). If out->tokens is NULL on entry, *out
 * receives device views of the tree inside the workspace, valid until the
 * next eagle_draft_tree; otherwise the tree is copied (on the stream) into
 * the caller's four arrays, which must hold batch * n_nodes+1 rows. */
eagle_status eagle_draft_tree(eagle_ctx* ctx, eagle_tree* out);

/* Verify ([LPD] "How EAGLE works": tree attention scores every node in one
 * forward pass): target pass over tree->n_rows rows per sequence at positions
 * L + depth, K/V written to slots L + row. d_argmax [batch][n_rows] receives the
 * greedy token after each row; d_logits [batch][n_rows][vocab] float32 receives
 * the logits when not NULL (debug/parity path). The tree may be the one
 * eagle_draft_tree returned or any caller-built tree (n_rows <= 121). The tree
 * is checked on the device against the rules stated at eagle_tree: a tree
 * that breaks one sets the device status, nothing is committed by the
 * following eagle_accept_commit, and the next eagle_sync_status returns
 * EAGLE_ERR_INVALID_ARG (the context is then spent). */
eagle_status eagle_verify(eagle_ctx* ctx, const eagle_tree* tree, int32_t* d_argmax, float* d_logits);

/* Accept and commit ([SDE] "Deep dive": longest correct prefix): greedy walk
 * over the last verified tree, compaction of the accepted K/V to contiguous
 * slots, features kept for the next draft. An accepted path longer than the
 * configured tree depth (a caller-built tree) is not cut short: nothing is
 * committed, *d_accept_len is -1 and the device status reports
 * EAGLE_ERR_INVALID_ARG. d_accept_len [batch] (may be NULL)
 * receives the accepted draft length a; d_tokens_out [batch][EAGLE_MAX_DEPTH+1]
 * (may be NULL) the a+1 committed tokens (accepted nodes, then the bonus token),
 * padded with -1. */
eagle_status eagle_accept_commit(eagle_ctx* ctx, int32_t* d_accept_len, int32_t* d_tokens_out);

/* Speculative generation ([SDE] "Deep dive": draft a tree, verify it in one
 * target pass, keep the longest correct prefix, repeat; the output equals the
 * target's own greedy decoding): prefill, then draft/verify/accept steps until
 * every sequence has at least max_new committed tokens (the prefill's first
 * token counts); d_out [batch][max_new] receives exactly max_new tokens per
 * sequence. With use_graph != 0 the step is captured once in a CUDA graph and
 * replayed. h_stats (may be NULL) is filled after the final synchronisation. */
eagle_status eagle_generate(eagle_ctx* ctx, const int32_t* d_prompt, int32_t prompt_len, int32_t max_new,
                            int32_t use_graph, int32_t* d_out, eagle_stats* h_stats);

/* Vanilla greedy decoding with the same kernels (one-row tree per step), the
 * lossless reference ([SDE] "Deep dive"). Same arguments as eagle_generate. */
eagle_status eagle_generate_vanilla(eagle_ctx* ctx, const int32_t* d_prompt, int32_t prompt_len,
                                    int32_t max_new, int32_t use_graph, int32_t* d_out, eagle_stats* h_stats);

/* Enqueue n_steps further steps (draft, verify, accept/commit; vanilla != 0:
 * one-row trees, i.e. plain greedy decoding) on a prefilled context without
 * any host synchronisation. With use_graph != 0 and a non-NULL stream, the
 * step is captured once into a CUDA graph (cached in the context) and
 * replayed. The caller keeps the KV capacity in mind: each step commits
 * between 1 and depth+1 tokens per sequence. */
eagle_status eagle_step(eagle_ctx* ctx, int32_t n_steps, int32_t vanilla, int32_t use_graph);

/* Kernel launches in one captured step (the CUDA graph's kernel nodes), or -1
 * before the first graph-captured eagle_step / eagle_generate. Host-only. */
int32_t eagle_step_kernel_count(const eagle_ctx* ctx, int32_t vanilla);

/* Synchronise the stream and return the device status word (EAGLE_OK if clean). */
eagle_status eagle_sync_status(eagle_ctx* ctx);

/* Copy the committed-token count per sequence (int32 [batch]) to device memory d_counts (on the stream). */
eagle_status eagle_committed_counts(eagle_ctx* ctx, int32_t* d_counts);

eagle_status eagle_destroy(eagle_ctx* ctx);
const char* eagle_last_error(const eagle_ctx* ctx);

/* sizeof of the ABI structs, for bindings to check their own layouts against:
 * which = 0 eagle_config, 1 eagle_weights, 2 eagle_layer_weights, 3 eagle_tree,
 * 4 eagle_stats; 0 for any other value. Host-only. */
size_t eagle_struct_size(int32_t which);

/* Weight-only int4 projections (config.weight_bits = 4). Input: a weight [N, K]
 * as 4-bit codes, row-major, two per byte (byte (n, i) holds code (n, 2i) in its
 * low and code (n, 2i + 1) in its high nibble; d_codes [N][K/2]) and bf16 scales
 * (d_scales [N][K/64], scale of row n and inputs 64g .. 64g+63); the weight is
 * W(n, k) = bf16(s(n, k/64) * (u(n, k) - 8)). eagle_int4_pack writes the layout
 * the kernels stream: blocks of 128 rows x 64 inputs, block (t, g) at byte
 * ((t K/64) + g) 4352, each 128 rows of 32 code bytes (word c of a row: input
 * 8c + 2i in bits 4i..4i+3 and 8c + 2i + 1 in bits 16+4i..19+4i) followed by the
 * 128 rows' scales. Needs N % 128 == 0 and K % 64 == 0 (else
 * EAGLE_ERR_UNSUPPORTED, and eagle_int4_packed_bytes returns 0); d_out (16-byte
 * aligned, eagle_int4_packed_bytes(N, K) bytes) is caller-owned. Asynchronous on
 * `stream`; the inputs may be freed once the stream has passed the call. For a
 * wqkv or wgu weight, pack the rows in the order of the bf16 layout (q, k, v rows;
 * gate / up rows interleaved in blocks of 64). */
size_t eagle_int4_packed_bytes(int32_t N, int32_t K);
eagle_status eagle_int4_pack(const uint8_t* d_codes, const uint16_t* d_scales, int32_t N, int32_t K, void* d_out,
                             void* stream);

/* ---------------------------------------------------------------------------
 * Kernel-level entry points: one hot-path kernel on caller buffers, for unit
 * parity tests and roofline timing. They run on `stream`, allocate nothing,
 * and need no context.
 * ------------------------------------------------------------------------- */

/* Y[M,N] (float32, row-major) = (X + X_lo)[M,K] W[N,K]^T with the verify-pass
 * GEMM kernel for `dtype` (bf16: tcgen05 + TMA weight streaming; f32: SIMT).
 * d_x_lo (bf16 only, may be NULL) holds the low halves of activations carried
 * as hi/lo bf16 pairs, as the step's GEMMs do.
 * N multiple of 128 and K multiple of 64 for bf16; X and W 16-byte aligned.
 * d_scratch (scratch_bytes >= eagle_op_gemm_scratch_bytes(M,N,K,dtype), else
 * EAGLE_ERR_WORKSPACE) holds split-K arrival counters and partial sums; the
 * caller zeroes it once, every launch leaves the counters at zero, and one
 * buffer sized for the largest shape serves every smaller one. Calls that
 * share a scratch buffer must not overlap on the GPU. */
size_t eagle_op_gemm_scratch_bytes(int32_t M, int32_t N, int32_t K, int32_t dtype);
eagle_status eagle_op_gemm(int32_t dtype, int32_t M, int32_t N, int32_t K, const void* d_x, const void* d_x_lo,
                           const void* d_w, float* d_y, void* d_scratch, size_t scratch_bytes, void* stream);

/* The same bf16 GEMM for callers that cannot allocate device memory: a plugin
 * inside a host framework that owns the device allocator and does not let its
 * plugins call cudaMalloc, or code whose device-memory budget is fixed by
 * someone else and has no room for a scratch buffer of its own. For them the
 * split-K scratch lives in a static device
 * array inside this library (10.5 MiB, reserved on every GPU that loads the
 * library until the process exits), so the caller passes only X, W and Y.
 * The pages have no counterpart; this is an interface convenience.
 *   - M <= 64 token rows, N a multiple of 128, K a multiple of 64; larger
 *     shapes return EAGLE_ERR_UNSUPPORTED (use eagle_op_gemm with a scratch).
 *   - Calls no cudaMalloc/cudaFree or allocating routine. The first call on a
 *     device looks up the array's device address (cudaGetSymbolAddress) with
 *     that device current; make that first call before any stream capture.
 *   - Every call shares the one array and clears the counters it uses before
 *     launching; calls that overlap on the GPU (other streams, other threads)
 *     race on it and must be serialised by the caller.
 *   - There is no status word: if one of the kernel's bounded waits gives up
 *     (2 s), the call has still returned EAGLE_OK and d_y is incomplete. */
eagle_status eagle_op_gemm_noalloc(int32_t M, int32_t N, int32_t K, const void* d_x, const void* d_w, float* d_y,
                                   void* stream);

/* Dense weights from eagle_int4_pack's layout: d_out [N][K] of `dtype` (f32 or
 * bf16) = bf16(scale * (code - 8)), the values every int4 GEMM of the library
 * multiplies with (the per-operation path expands them like this; the persistent
 * kernel expands each block in shared memory). Asynchronous on `stream`. */
eagle_status eagle_op_int4_dequant(const void* d_w4, int32_t N, int32_t K, int32_t dtype, void* d_out,
                                   void* stream);

/* The same products run by the persistent layer-stack kernel (the kernel of the
 * verify and draft passes), for checking its work split against eagle_op_gemm
 * and eagle_op_lmhead_topk: n_phases GEMM phases Y = (X + X_lo) W^T in one
 * cooperative launch, each waiting for the previous one. k == 0: every phase
 * stores Y into d_y. k > 0: the last phase is the LM-head epilogue instead
 * (top-k per row, merged into d_idx/d_val/d_lse as eagle_op_lmhead_topk does;
 * d_val and d_lse may be NULL). bf16 only; 1 <= M <= 128, N % 128 == 0,
 * K % 64 == 0, k <= 16. d_scratch: eagle_op_gemm_persistent_scratch_bytes()
 * bytes, zeroed once before first use (the kernel leaves its counters zero).
 * Synchronises `stream` before returning. */
size_t eagle_op_gemm_persistent_scratch_bytes(int32_t M, int32_t N, int32_t K, int32_t n_phases, int32_t k);
eagle_status eagle_op_gemm_persistent(int32_t M, int32_t N, int32_t K, int32_t n_phases, int32_t k,
                                      const void* d_x, const void* d_x_lo, const void* d_w, float* d_y,
                                      int32_t* d_idx, float* d_val, float* d_lse, void* d_scratch,
                                      size_t scratch_bytes, void* stream);

/* LM head + per-row top-k: for each row m of X [M,K], the k largest logits of
 * X W^T (W [N,K]) as (index, value) ordered by value desc then index asc, and
 * the row's log-sum-exp. d_idx/d_val [M][k], d_lse [M]. */
size_t eagle_op_lmhead_scratch_bytes(int32_t M, int32_t N, int32_t K, int32_t k, int32_t dtype);
eagle_status eagle_op_lmhead_topk(int32_t dtype, int32_t M, int32_t N, int32_t K, int32_t k, const void* d_x,
                                  const void* d_w, int32_t* d_idx, float* d_val, float* d_lse, void* d_scratch,
                                  size_t scratch_bytes, void* stream);

/* Tree attention for one sequence over a KV cache slice: queries Q [rows][n_heads][hd]
 * (float32, RoPE applied), keys/values K,V [n_kv_heads][cap][hd] (the KV-cache type of dtype:
 * float32 for EAGLE_DTYPE_F32, IEEE half for EAGLE_DTYPE_BF16); row r attends to slots
 * [0, prefix) and to slot prefix + i of the tree block for each bit i set in
 * mask[r] (two uint64 words). Output O [rows][n_heads][hd] (dtype elements). */
size_t eagle_op_attention_scratch_bytes(int32_t rows, int32_t n_heads, int32_t hd, int32_t prefix);
eagle_status eagle_op_tree_attention(int32_t dtype, int32_t rows, int32_t n_heads, int32_t n_kv_heads,
                                     int32_t hd, int32_t cap, int32_t prefix, const void* d_q, const void* d_k,
                                     const void* d_v, const uint64_t* d_mask, void* d_o, void* d_scratch,
                                     size_t scratch_bytes, void* stream);

/* Phase trace of the verify pass (profiling aid; no counterpart in the pages).
 * On a bf16 context whose verify pass runs as one persistent launch, reports
 * that program's phase count P (per layer: QKV, attention, merge, O, gate/up,
 * down; then the LM head) and the CTA count C; either output may be NULL.
 * With d_trace non-NULL (device memory of n >= (P + 1) * C uint64 words, owned
 * by the caller and kept alive while set), every later verify launch writes
 * d_trace[p * C + c] = %globaltimer (ns) when CTA c finished phase p, and
 * d_trace[P * C + c] = when CTA c started. d_trace NULL turns tracing off.
 * EAGLE_ERR_INVALID_ARG if n is too small or the context has no persistent
 * verify pass (then P = C = 0). Drops any captured step graph. */
eagle_status eagle_set_trace(eagle_ctx* ctx, uint64_t* d_trace, size_t n, int32_t* n_phases, int32_t* n_ctas);

/* Failure-detection self-test (no counterpart in the pages): one GPU thread
 * waits, with the same bounded wait as the GEMM pipeline's mbarrier waits, on
 * a barrier that nothing arrives on. After the wait's time limit (2 s) it gives
 * up, writes EAGLE_ERR_TIMEOUT to *d_status (if *d_status was EAGLE_OK) and the
 * kernel returns; no trap, no fault, and the CUDA context stays usable. */
eagle_status eagle_selftest_bounded_wait(int32_t* d_status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* EAGLE_H */
