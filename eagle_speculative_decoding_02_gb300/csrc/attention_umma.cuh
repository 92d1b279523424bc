// Tree-masked attention work item on the 5th-generation tensor cores
// (tcgen05.mma, operands in shared memory, scores and output in tensor memory),
// run by the four epilogue warps of the persistent layer-stack kernel, and by
// the standalone items / merge launches of attention_umma.cu.
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
//   5. The row's unnormalised partial (O, max, sum) goes out for the merge
//      (PartLayout). The next item's copies are issued as soon as the MMAs are
//      done, so they overlap this step.
//
// Precision: half q, K, P and V, fp32 accumulation.
#pragma once

#include "attention_common.cuh"
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
  const Group* groups; // the launch's attention groups (a copy in shared memory)
  uint32_t kv_par = 0, mma_par = 0;
};

// Balanced split of a group's keys. A group's rows see the slots [0, T),
// T = prefix + block_len: the prefix (every key visible) and then the tree block
// (keys seen through the ancestor masks). The slots are cut into parts of
// ps <= 128 keys: ns = max(n0, ceil(T / 128)) parts requested, where n0 = the
// CTAs per (KV head, row tile) pair of the whole phase, ps = ceil(T / ns), and
// ceil(T / ps) non-empty parts result. With every part of equal size and, when
// the keys allow it, no more items than CTAs, no CTA runs two items while
// others wait (128-key chunks plus the tree block gave 160 items for 152 CTAs
// at a 1040-key prefix). Part j covers slots [j ps, min((j + 1) ps, T)).
__device__ __forceinline__ int um_part_keys(const Group& g, int n0) {
  const int T = g.prefix + g.block_len;
  const int ns = max(n0, (T + kUmKeys - 1) / kUmKeys);
  return max(1, (T + ns - 1) / ns);
}
__device__ __forceinline__ int um_parts(const Group& g, int n0) {
  const int T = g.prefix + g.block_len;
  const int ps = um_part_keys(g, n0);
  return (T + ps - 1) / ps;
}

// Partial slots per row that any phase may need: ceil(T / 128) <= the chunk
// count of the longest prefix, and n0 <= max_ctas / Hkv.
__host__ __device__ inline int um_part_slots(int max_prefix, int Hkv, int max_ctas) {
  const int a = n_prefix_chunks(max_prefix, kUmKeys), b = max_ctas / Hkv;
  return (a > b ? a : b) + 1;
}

// Bits off .. off + 31 of the 128-bit value (hi:lo), zero outside bits [0, 128).
__device__ __forceinline__ uint32_t bits32(uint64_t lo, uint64_t hi, int off) {
  if (off <= -32 || off >= 128) return 0u;
  if (off < 0) return (uint32_t)(lo << (-off));
  if (off == 0) return (uint32_t)lo;
  if (off < 64) return (uint32_t)((lo >> off) | (hi << (64 - off)));
  return (uint32_t)(hi >> (off - 64));
}

// An item: part of the group's keys, KV head, 128-row tile, group.
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
                         const CUtensorMap* tmV, const UmItem& it, int n0, const UmState& st) {
  const int Hq = a.Hq, Hkv = a.Hkv, Mrows = a.M, cap = a.cap;
  const Group g = st.groups[it.z];
  const int G = Hq / Hkv;
  const int key0 = it.chunk * um_part_keys(g, n0);
  uint8_t* sQ = st.sm;
  uint8_t* sV = sQ + (size_t)kUmRows * HD * 2;
  uint8_t* sK = sV + (size_t)kUmKeys * HD * 2;
  // q and this layer's new K / V rows were written by other SMs' generic stores
  // earlier in the launch; the copies read them through the async proxy
  asm volatile("fence.proxy.async.global;" ::: "memory");
  mbar_expect_tx(st.kv_bar, (uint32_t)(3 * kUmRows * HD * 2));
  const int ykv = (g.seq * Hkv + it.kvh) * cap + key0;
  const int yq = (it.kvh * Mrows + g.row0) * G + it.rt * kUmRows;
#pragma unroll
  for (int h = 0; h < HD / 64; ++h) {
    tma_load_2d(sQ + h * kUmAtom, tmQ, st.kv_bar, h * 64, yq);
    tma_load_2d(sK + h * kUmAtom, tmK, st.kv_bar, h * 64, ykv);
    tma_load_2d(sV + h * kUmAtom, tmV, st.kv_bar, h * 64, ykv);
  }
}

// The attention work items that have keys and rows, in order (group, KV head,
// 128-row tile, part of the keys): count() counts them, item() decodes one. The
// keys of every group are split into parts by the balanced rule of
// um_part_keys, with n0 = the CTAs per (KV head, row tile) pair.
struct UmItems {
  const Group* groups;  // the phase's groups (shared-memory copy)
  int n_groups, Hkv, G;  // (copied: the arguments live in global memory)
  int n0 = 1;
  __device__ UmItems(const AttnArgs& a, const Group* g, int n_ctas)
      : groups(g), n_groups(a.n_groups), Hkv(a.Hkv), G(a.Hq / a.Hkv) {
    int pairs = 0;
    for (int z = 0; z < n_groups; ++z) pairs += Hkv * rts(groups[z]);
    n0 = pairs > 0 ? max(1, n_ctas / pairs) : 1;
  }
  __device__ int rts(const Group& g) const { return um_row_tiles(g.nrows, G); }
  __device__ int chunks(const Group& g) const { return um_parts(g, n0); }
  __device__ int count() const {
    int n = 0;
    for (int z = 0; z < n_groups; ++z) {
      const Group g = groups[z];
      n += chunks(g) * Hkv * rts(g);
    }
    return n;
  }
  __device__ void item(int i, int& chunk, int& kvh, int& rt, int& z) const {
    for (z = 0; z < n_groups; ++z) {
      const Group g = groups[z];
      const int nc = chunks(g), nr = rts(g), n = nc * Hkv * nr;
      if (i < n) {
        chunk = i % nc;
        const int rest = i / nc;
        kvh = rest / nr;
        rt = rest % nr;
        return;
      }
      i -= n;
    }
    chunk = kvh = rt = z = 0;
  }
};

// One item, run by 128 threads: tid 0..127 (tid 0 issues the copies and MMAs),
// row = the TMEM lane this thread may read (its warp's lane quarter x 32 + lane)
// and thus its row of the tile. sync() is a barrier over the 128 threads. The
// item's copies were issued (um_issue); once its MMAs are done and before its
// partials go out, thread 0 issues those of `next` when has_next. The caller
// passes only items with keys and rows; n0 is the phase's parts request (see
// um_part_keys). Returns false on a timeout (status set, abort raised).
template <int HD, typename Sync>
__device__ bool attn_item_um(const AttnArgs& a, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                             const CUtensorMap* tmV, const UmItem& cur, bool has_next, const UmItem& next,
                             int n0, int n_chunk_slots, UmState& st, int tid, int row, volatile int* abort_flag,
                             Sync sync) {
  static_assert(HD == 64 || HD == 128, "head dim");
  // the arguments live in global memory: read them once into registers (the
  // partial stores below could otherwise force reloads)
  const int Hq = a.Hq, Hkv = a.Hkv, Mrows = a.M;
  const uint64_t* const mask = a.mask;
  float* const part = a.part;
  int* const status = a.status;
  const Group g = st.groups[cur.z];
  const int G = Hq / Hkv;
  const int R = g.nrows * G;
  const int ps = um_part_keys(g, n0);
  const int key0 = cur.chunk * ps;                                  // the box's first slot
  const int nkeys = min(ps, g.prefix + g.block_len - key0);         // this part's keys
  const int r = cur.rt * kUmRows + row;
  const bool rv = r < R;
  const int node = rv ? r / G : 0;
  const int qh = cur.kvh * G + (rv ? r % G : 0);
  uint8_t* sQ = st.sm;
  uint8_t* sV = sQ + (size_t)kUmRows * HD * 2;
  uint8_t* sK = sV + (size_t)kUmKeys * HD * 2;  // K, then P
  const uint32_t lane_base = (uint32_t)(row & ~31) << 16;

  // visibility of this row's keys, 32 per word: box row i (slot key0 + i) is
  // visible when i < nkeys and the slot is in the prefix, or is tree-block slot
  // prefix + t with bit t set in the node's ancestor mask
  uint32_t vis[kUmKeys / 32];
  {
    uint64_t mk0 = 0ull, mk1 = 0ull;
    if (rv && key0 + nkeys > g.prefix) {
      mk0 = mask[2 * (g.row0 + node)];
      mk1 = mask[2 * (g.row0 + node) + 1];
    }
    const int npre = g.prefix - key0;  // box rows below the tree block
#pragma unroll
    for (int b = 0; b < kUmKeys / 32; ++b) {
      const int nv = nkeys - 32 * b, np = npre - 32 * b;
      const uint32_t valid = nv >= 32 ? ~0u : (nv <= 0 ? 0u : (1u << nv) - 1u);
      const uint32_t pre = np >= 32 ? ~0u : (np <= 0 ? 0u : (1u << np) - 1u);
      const uint32_t blk = bits32(mk0, mk1, key0 + 32 * b - g.prefix);
      vis[b] = rv ? (valid & (pre | blk)) : 0u;
    }
  }

  // 1. S = Q K^T once the copies have landed
  bool ok = true;
  if (tid == 0) {
    ok = mbar_wait(st.kv_bar, st.kv_par, abort_flag, status);
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
  if (ok) ok = epi_all(mbar_wait(st.mma_bar, st.mma_par, abort_flag, status));
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
  ok = epi_all(mbar_wait(st.mma_bar, st.mma_par, abort_flag, status));
  st.mma_par ^= 1;
  if (!ok) return false;
  tc_fence_after();
  // every tile is free again: the next item's copies overlap this item's output
  if (tid == 0 && has_next) um_issue<HD>(a, tmQ, tmK, tmV, next, n0, st);

  // 4. the row's partial (tcgen05.ld is warp-wide: every lane loads)
  const PartLayout pl{part, Mrows * Hq, n_chunk_slots, HD};
  const int w = (g.row0 + node) * Hq + qh;
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

// The group holding verify row `row` (the groups partition the rows).
__device__ __forceinline__ int um_group_of(const Group* groups, int n_groups, int row) {
  for (int z = 0; z < n_groups; ++z)
    if (row >= groups[z].row0 && row < groups[z].row0 + groups[z].nrows) return z;
  return -1;  // a padding row: in no group, no item wrote its partials
}

// Merge of the persistent kernel over this CTA's (row, query head) pairs
// w in [w0, w1): the combination of each pair's part partials (max, sum,
// unnormalised output) in part order (a running maximum, the flash-decoding combination), with the
// partials staged in shared memory first. For every part s and 32-column block,
// the partials of consecutive pairs are contiguous in the partial buffer, so a
// few bulk copies bring all of them in one round trip (instead of dozens of
// dependent loads per pair, which made this phase latency-bound); the (max, sum)
// pairs come by plain loads. Parts are taken in batches that fit `sm_bytes` of
// shared memory at `sm`, with each pair's running (max, sum, output) kept there
// between batches. Run by the 128 epilogue threads; bar = an mbarrier of this
// CTA with parity *par. Returns false on a timeout.
template <int HD, typename Sync>
__device__ bool um_merge_staged(const AttnArgs& a, const Group* groups, int n0, int w0, int w1, int n_chunk_slots,
                                uint8_t* sm, uint32_t sm_bytes, uint64_t* bar, uint32_t* par, int tid,
                                volatile int* abort_flag, Sync sync) {
  const int nw = w1 - w0;
  if (nw <= 0) return true;
  constexpr int NB = HD / 32;
  // the arguments live in global memory: read them once into registers (the
  // output stores below could otherwise force a reload after each of them)
  const int Hq = a.Hq, n_groups = a.n_groups;
  bf16* const out = reinterpret_cast<bf16*>(a.o);
  bf16* const out_lo = a.o_lo;
  int* const status = a.status;
  const PartLayout pl{a.part, a.M * Hq, n_chunk_slots, HD};
  const int ew = tid >> 5, lane = tid & 31;
  float* run = reinterpret_cast<float*>(sm);  // [nw][HD + 2]: running output, then (max, sum)
  const uint32_t run_bytes = ((uint32_t)nw * (HD + 2) * 4 + 127) & ~127u;
  uint8_t* stage = sm + run_bytes;
  const uint32_t per_part = (uint32_t)nw * (HD * 4 + 8);
  const int sb = run_bytes + per_part <= sm_bytes ? (int)((sm_bytes - run_bytes) / per_part) : 0;
  if (sb < 1) {
    set_status(status, kStCapacity);
    return false;
  }
  // the most parts any of these pairs' groups has
  const int r0 = w0 / Hq, r1 = (w1 - 1) / Hq;
  int nmax = 0;
  for (int z = 0; z < n_groups; ++z) {
    const Group g = groups[z];
    if (g.row0 <= r1 && g.row0 + g.nrows > r0) nmax = max(nmax, um_parts(g, n0));
  }
  for (int s0 = 0; s0 < nmax; s0 += sb) {
    const int ns = min(sb, nmax - s0);
    float2* mls = reinterpret_cast<float2*>(stage + (size_t)ns * NB * nw * 128);  // [ns][nw]
    // thread 0 announces the bytes, then the copies are issued by as many
    // threads (a transaction count may run ahead of its announcement)
    if (tid == 0) mbar_expect_tx(bar, (uint32_t)ns * NB * nw * 128);
    // the partials were written by other SMs' generic stores earlier in the launch
    asm volatile("fence.proxy.async.global;" ::: "memory");
    for (int i = tid; i < ns * NB; i += 128)
      bulk_load(stage + (size_t)i * nw * 128, pl.o(s0 + i / NB, w0, i % NB), (uint32_t)nw * 128, bar);
    for (int i = tid; i < ns * nw; i += 128) {
      const int s = i / nw, t = i - s * nw;
      mls[i] = __ldcg(reinterpret_cast<const float2*>(pl.ml(s0 + s, w0 + t)));
    }
    sync();
    const bool ok = epi_all(mbar_wait(bar, *par, abort_flag, status));
    *par ^= 1;
    if (!ok) return false;
    const float* os = reinterpret_cast<const float*>(stage);
    for (int t = ew; t < nw; t += 4) {
      const int w = w0 + t, row = w / Hq, qh = w - row * Hq;
      // a padding row (in no group) has no parts: its output is zero, not a mix of stale partials
      const int z = um_group_of(groups, n_groups, row);
      const int nck = z >= 0 ? um_parts(groups[z], n0) : 0;
      float M = -INFINITY, L = 0.f, acc[NB];
      if (s0 == 0) {
#pragma unroll
        for (int i = 0; i < NB; ++i) acc[i] = 0.f;
      } else {
#pragma unroll
        for (int i = 0; i < NB; ++i) acc[i] = run[(size_t)t * (HD + 2) + NB * lane + i];
        M = run[(size_t)t * (HD + 2) + HD];
        L = run[(size_t)t * (HD + 2) + HD + 1];
      }
      const int se = min(s0 + ns, nck);
      // kJ parts at a time with no branch: every load reads a valid slot (the
      // index is clamped) and parts past se weigh zero, so all the loads of a
      // batch are independent and issue together (one part after another would
      // be a chain of dependent loads and branches on one warp per scheduler).
      // kJ = 10 takes the 9-10 parts of a bs-1 verify at a 1-1.2k-token prefix in
      // one batch (8 took two: merge phase 8.5 -> 8.0 us per layer)
      constexpr int kJ = 10;
      for (int sj = s0; sj < se; sj += kJ) {
        float mm[kJ], ll[kJ], ov[kJ][NB];
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
          const int sl = min(sj + j, se - 1) - s0;
          const float2 ml = mls[sl * nw + t];
          mm[j] = sj + j < se ? ml.x : -INFINITY;
          ll[j] = ml.y;
          // this lane's NB neighbouring columns NB lane .. NB lane + NB - 1: one vector
          // load, and the output below is one store of NB neighbours (one column in
          // every 32-column block took NB loads and 2 NB stores: merge phase 7.9 ->
          // 7.2 us per layer of the 8B verify)
          const float* src = os + (((size_t)sl * NB + (NB * lane) / 32) * nw + t) * 32 + (NB * lane) % 32;
          if constexpr (NB == 4) {
            const float4 v4 = *reinterpret_cast<const float4*>(src);
            ov[j][0] = v4.x; ov[j][1] = v4.y; ov[j][2] = v4.z; ov[j][3] = v4.w;
          } else {
#pragma unroll
            for (int i = 0; i < NB; ++i) ov[j][i] = src[i];
          }
        }
        float Mb = M;
#pragma unroll
        for (int j = 0; j < kJ; ++j) Mb = fmaxf(Mb, mm[j]);
        const float Ms = Mb == -INFINITY ? 0.f : Mb;  // (every weight is 0 then)
        const float r = M == -INFINITY ? 0.f : exp2f(M - Ms);
        L *= r;
#pragma unroll
        for (int i = 0; i < NB; ++i) acc[i] *= r;
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
          const float wgt = exp2f(mm[j] - Ms);  // exp2(-inf) = 0 for masked parts
          L += wgt * ll[j];
#pragma unroll
          for (int i = 0; i < NB; ++i) acc[i] += wgt * ov[j][i];
        }
        M = Mb;
      }
      if (s0 + ns >= nmax) {
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const size_t ob = ((size_t)row * Hq + qh) * HD;
        if constexpr (NB == 4) {
          store_hilo4<bf16>(out, out_lo, ob + 4 * lane,
                            make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv));
        } else {
#pragma unroll
          for (int i = 0; i < NB; ++i) store_hilo<bf16>(out, out_lo, ob + NB * lane + i, acc[i] * inv);
        }
      } else {
#pragma unroll
        for (int i = 0; i < NB; ++i) run[(size_t)t * (HD + 2) + NB * lane + i] = acc[i];
        if (lane == 0) {
          run[(size_t)t * (HD + 2) + HD] = M;
          run[(size_t)t * (HD + 2) + HD + 1] = L;
        }
      }
    }
    // this batch's staging is read: the next batch's copies may overwrite it
    fence_proxy_async_smem();
    sync();
  }
  return true;
}

}  // namespace attn
}  // namespace eg
