// Persistent layer-stack forward on the sm_103a tensor cores (tcgen05 + TMA).
//
// At one verify or draft step of EAGLE ("EAGLE (LLM decoding)", section "How
// EAGLE works") every decoder layer multiplies a few dozen token rows by its
// weight matrices: each GEMM is a 5-35 us stream of weights, and as separate
// kernels each pays a launch, a pipeline fill and a split-K tail. Here one
// cooperative launch (one CTA per SM) runs the whole program of phases:
//
//   GEMM   swap-AB tcgen05 tiles (128 weight rows x MT token rows, fp32 in TMEM),
//          (tile, 64-wide k-block) units: whole tiles dealt to every CTA, the
//          remainder split evenly over the CTAs (stream-K) and run first,
//          split tiles summed at the end of the phase by all their CTAs, each a
//          slice of the rows, in ascending CTA order,
//          then the fused epilogue (RMSNorm row scale, RoPE + KV write, SwiGLU,
//          residual add + next norm, LM-head top-k records).
//   ATTN   tree-attention work items (128-key chunk, KV head, 128-row tile,
//          group) on the same tensor cores (attention_umma.cuh), run by the
//          epilogue warps with S and O in tensor memory, partials to global memory.
//   MERGE  one warp per (row, query head) combines the partials in chunk order.
//
// Phase p reads only what phases < p wrote. A CTA that has finished all its
// epilogue work of phase p adds one to counter done[p] (release); consumers of
// phase p wait until it reaches the grid size (acquire). Weight boxes depend on
// nothing, so the weight producer streams the weights of later GEMM phases into
// its ring while earlier phases finish; only the activation boxes of phase p
// wait for done[p - 1].
//
// Warp roles (224 threads):
//   warp 0     weight producer (one lane): weight half of each ring slot
//   warp 1     TMEM allocator and MMA issuer (one lane)
//   warps 2-5  epilogue, attention and merge (128 threads)
//   warp 6     activation producer (one lane): activation half of each ring slot
// Unit i uses ring slot i % S in both halves; one full barrier per slot takes
// both producers' arrivals and bytes, one empty barrier (the MMA's commit)
// frees the slot for both, as in a single-producer pipeline.
// Weight-only int4 programs (a GEMM phase whose weight is a packed int4 block
// array, int4.cuh) run a variant with 352 threads: warp 0 streams the packed
// blocks (4352 bytes per 128 x 64 unit) through a deeper ring of their own, and
// converter warps 7-10 (32 weight rows each) expand each block to the bf16 slot
// layout above (the TMA's 128-byte swizzle) once the MMA has freed the slot;
// they also issue the bf16 boxes of the program's 16-bit phases. A slot's full
// barrier then takes the activation producer's and the unit's converter warp's
// arrivals. (A separate, deeper activation ring was measured: no gain; the
// MMA issue loop, one thread at ~900 cycles per unit, is what limits this
// variant at 61 rows.)
// Every wait is bounded (2 s); on a timeout the CTA records kStTimeout, stops
// issuing work, drains its copies and returns; other CTAs then time out on
// their own waits.
#include <cuda.h>

#include "../../include/eagle.h"
#include "attention_common.cuh"
#include "attention_umma.cuh"
#include "epilogue.cuh"
#include "int4.cuh"
#include "stack.h"
#include "tc_ptx.cuh"
#include "topk.cuh"

namespace eg {
namespace {

using namespace tc;

constexpr int kThreads = 224;
constexpr int kThreadsW4 = 352;            // int4 variant: + converter warps 7-10
constexpr int kConvWarp = 7;
constexpr int kMaxRaw = 32;                // int4 variant: packed-block ring stages (upper bound)
constexpr int kXWarp = 6;                  // activation producer warp
constexpr int kBK = 64;
constexpr int kWBytes = kTileN * kBK * 2;  // 16 KB weight box
constexpr int kSub = 32;                   // epilogue rows per sub-tile
constexpr int kLdt = kTileN + 4;  // rows 16-byte aligned for the epilogues' vector accesses
constexpr int kMaxW = 12;                  // weight ring stages (upper bound)
constexpr int kAttnCKI = attn::kUmKeys;    // keys per attention work item
constexpr int kSmemBudget = 232448;        // 227 KB opt-in per block
constexpr int kMaxCtas = 160;              // partial buffer sizing bound
constexpr int kEpiThreads = 128;           // epilogue warps 2-5
constexpr int kMaxGroups = 128;            // attention groups kept in shared memory
// epilogue staging: one sub-tile, then the row inputs of every row of the phase
constexpr size_t kTileBytes = (size_t)(kSub * kLdt + 4 * kStackMaxRows) * 4;

struct StackArgs {
  const StackPhase* ph;
  int n_phases;
  int M, MT, has_lo, sw, sx;
  int rw;            // int4 variant: packed-block ring stages
  int apad;          // bytes after the epilogue tile that complete the attention staging region
  uint32_t tmem_cols;
  unsigned* done;    // [n_phases] phase counters, then the exit counter
  int* tile_cnt;     // [n_counters] split-K arrival counters
  int n_counters;
  float* partial;    // [G][2][MT][128]
  int* status;
  unsigned long long* trace;  // optional: [n_phases + 1][G] %globaltimer stamps
  float* y_last;              // optional: output y of the last phase's epilogue (LM-head logits)
  const Group* groups;        // attention groups of every attention phase (NULL if none)
  int n_groups;               // <= kMaxGroups
  int first_attn;             // index of the first attention phase, -1 if none (all share rows and groups)
  TopkMerge mg;               // mg.k > 0: merge of the last (LM-head) phase's records, CTA c taking row c
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

__device__ __forceinline__ long long unit_start(long long T, int c, int Gp) { return (long long)c * T / Gp; }
__device__ __forceinline__ int cta_of(long long T, long long u, int Gp) { return (int)(((u + 1) * Gp - 1) / T); }

// Work split of a GEMM phase of n_s tiles x kbt k-blocks over Ga of the G CTAs:
// every CTA owns Wd = n_s / Ga whole tiles (data-parallel); the R = n_s - Wd Ga
// remaining tiles are split stream-K over min(Ga, R kbt) CTAs. A CTA runs its
// split units first, so that the split tiles are summed while its whole tiles
// stream. Ga = G, except when the phase has fewer tiles than CTAs and a whole
// number k = G / n_s of CTAs per tile still covers kAlignPct percent of the grid:
// then Ga = k n_s, so that each tile is split over exactly k CTAs and no CTA's
// range crosses a tile boundary. A CTA then sums one split tile instead of two:
// the second sum and epilogue of the CTAs whose range crossed a boundary set
// these phases' ends. Measured on the 8B verify (152 CTAs): QKV (48 tiles, 144
// CTAs) 23.2 -> 19.2 us, O and down (32 tiles, 128 CTAs) 19.9 -> 15.7 and 29.5
// -> 26.6 us per layer, although a sixth of the grid then streams no weights.
constexpr int kAlignPct = 80;
struct Split {
  int kbt, Wd, Gs, Ga;
  long long Ts, base;  // split units, first split unit
  __device__ Split(const StackPhase& P, int G) {
    kbt = P.kbt;
    const int ns = P.n_tiles;
    Ga = G;
    if (ns < G && ns * (G / ns) * 100 >= kAlignPct * G) Ga = ns * (G / ns);
    Wd = ns / Ga;
    Ts = (long long)(ns - Wd * Ga) * kbt;
    base = (long long)Wd * Ga * kbt;
    Gs = Ts > 0 ? (int)min((long long)Ga, Ts) : 0;
  }
  __device__ void split_range(int c, int& u0, int& u1) const {
    if (c < Gs) {
      u0 = (int)(base + unit_start(Ts, c, Gs));
      u1 = (int)(base + unit_start(Ts, c + 1, Gs));
    } else {
      u0 = u1 = 0;
    }
  }
  __device__ void whole_range(int c, int& u0, int& u1) const {
    u0 = c < Ga ? c * Wd * kbt : 0;
    u1 = c < Ga ? u0 + Wd * kbt : 0;
  }
  // the CTAs c0..c1 that share split tile t
  __device__ void sharers(int t, int& c0, int& c1) const {
    const long long l0 = (long long)t * kbt - base;
    c0 = cta_of(Ts, l0, Gs);
    c1 = cta_of(Ts, l0 + kbt - 1, Gs);
  }
  // first tile of CTA cc's split range (its partial slot 0 holds that tile)
  __device__ int first_split_tile(int cc) const { return (int)((base + unit_start(Ts, cc, Gs)) / kbt); }
};

// This CTA's units [u, u1) of GEMM phase p, its split range (stage 0) then its
// whole tiles (stage 1); unit u is k-block kb of tile sl. next() moves to the
// next non-empty range; advance() steps one unit. The producer and MMA loops run
// on one thread each, so the per-unit bookkeeping avoids integer division.
struct Cursor {
  int p = -1, stage = 1;
  int u = 0, u1 = 0, kbt = 1, sl = 0, kb = 0;
  __device__ bool start(const StackArgs& a) {
    kbt = a.ph[p].kbt;
    sl = u / kbt;
    kb = u - sl * kbt;
    return true;
  }
  __device__ bool next(const StackArgs& a, int c, int G) {
    for (;;) {
      if (stage == 0) {
        stage = 1;
        Split(a.ph[p], G).whole_range(c, u, u1);
        if (u < u1) return start(a);
      }
      for (++p; p < a.n_phases && a.ph[p].kind != kPhaseGemm; ++p) {
      }
      if (p >= a.n_phases) return false;
      stage = 0;
      Split(a.ph[p], G).split_range(c, u, u1);
      if (u < u1) return start(a);
    }
  }
  // step n units within the current tile (kb + n <= kbt)
  __device__ bool advance(const StackArgs& a, int c, int G, int n = 1) {
    u += n;
    kb += n;
    if (kb == kbt) {
      kb = 0;
      ++sl;
    }
    return u < u1 || next(a, c, G);
  }
};

// Position in the ring: slot s of round r (the r-th pass over the S slots).
// A slot's full barrier completes once per round (parity r & 1); a producer
// refilling slot s in round r >= 1 waits for empty completion r - 1.
struct RingPos {
  int s = 0;
  uint32_t r = 0;
  __device__ void step(int S) {
    if (++s == S) {
      s = 0;
      ++r;
    }
  }
};

// Bounded wait until done[p] reaches G (one thread).
__device__ bool wait_phase(const StackArgs& a, int p, unsigned G, volatile int* abort_flag) {
  if (ld_acquire(a.done + p) >= G) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    __nanosleep(64);  // back off: the other warps of the SM keep working meanwhile
    if (ld_acquire(a.done + p) >= G) return true;
    if ((i & 15) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        set_status(a.status, kStTimeout);
        return false;
      }
    }
  }
}

// Bounded wait until split-K counter i reaches n (one thread).
__device__ bool wait_count(const StackArgs& a, int i, unsigned n, volatile int* abort_flag) {
  const unsigned* p = reinterpret_cast<const unsigned*>(a.tile_cnt + i);
  if (ld_acquire(p) >= n) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t k = 1;; ++k) {
    __nanosleep(64);
    if (ld_acquire(p) >= n) return true;
    if ((k & 15) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > kTimeoutNs) {
        *abort_flag = 1;
        set_status(a.status, kStTimeout);
        return false;
      }
    }
  }
}

template <int HD, bool W4>
__global__ void __launch_bounds__(W4 ? kThreadsW4 : kThreads, 1) stack_tc_kernel(StackArgs a) {
  constexpr int NT = W4 ? kThreadsW4 : kThreads;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned (128-byte swizzled TMA boxes) by an offset from the shared
  // array itself: a pointer rebuilt from an integer loses its address space, and
  // every access through it is then a generic one (measured: the merge phase 10.5
  // -> 8.7 us, the verify 4.16 -> 4.10 ms with shared-space accesses)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int S = a.sw, MT = a.MT;
  const int accw = a.has_lo ? 2 * MT : MT;  // accumulator columns of one tile
  const int abufw = accw;                   // accumulator columns of one buffer
  const int wslot = kWBytes;                // weight bytes of a ring slot
  const int xbox = MT * kBK * 2;
  const int xbytes = xbox * (a.has_lo ? 2 : 1);
  uint8_t* wring = smem;
  uint8_t* xring = wring + (size_t)S * wslot;
  float* tile = reinterpret_cast<float*>(xring + (size_t)S * xbytes);
  // Attention phases run while the activation halves and the epilogue tile are
  // idle (the next GEMM phase's boxes wait for them to finish), so their Q, K / P
  // and V tiles alias those (padded by apad bytes where they are too small).
  const EpiRows prow = epi_rows(tile + kSub * kLdt, kStackMaxRows);  // row inputs of the current GEMM phase
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(tile) + kTileBytes + a.apad);
  uint64_t* full = bars;
  uint64_t* empty = full + S;
  uint64_t* afull = empty + S;
  uint64_t* aempty = afull + 2;
  uint64_t* drain = aempty + 2;
  uint64_t* at_kv = drain + 1;   // attention: K / V copies
  uint64_t* at_mma = at_kv + 1;  // attention: S and O MMAs
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(at_mma + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = abort_flag + 1;
  volatile int* exit_last = abort_flag + 2;
  Group* sgroups = reinterpret_cast<Group*>(tmem_slot + 4);  // kMaxGroups entries
  // int4 variant: the packed-block ring and its barriers after the groups
  uint8_t* const rbase = reinterpret_cast<uint8_t*>(sgroups + kMaxGroups);
  uint64_t* rfull = reinterpret_cast<uint64_t*>(rbase + ((16u - (smem_u32(rbase) & 15u)) & 15u));
  uint64_t* rempty = rfull + a.rw;
  uint8_t* rraw = reinterpret_cast<uint8_t*>(rempty + a.rw);  // 16-byte aligned (2 rw barriers of 8 bytes)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, G = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 2);  // the activation producer, and the weight producer or the unit's converter warp
      mbar_init(&empty[s], 1);
    }
    if (W4)
      for (int j = 0; j < a.rw; ++j) {
        mbar_init(&rfull[j], 1);   // the packed-block producer (transaction bytes)
        mbar_init(&rempty[j], 1);  // the unit's converter warp, once read
      }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&afull[b], 1);
      mbar_init(&aempty[b], 4);
    }
    mbar_init(drain, 1);
    mbar_init(at_kv, 1);
    mbar_init(at_mma, 1);
    *abort_flag = 0;
    *last_flag = 0;
    *exit_last = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the groups of the attention phases, read once (the item loops decode them often)
  for (int i = threadIdx.x; i < a.n_groups; i += NT) sgroups[i] = a.groups[i];
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(a.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (a.trace && threadIdx.x == 0) a.trace[(size_t)a.n_phases * G + c] = globaltimer();

  if (W4 && warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ packed-block producer (int4 variant)
      // The int4 phases' blocks stream into their own ring, ahead of the
      // conversions; units of 16-bit phases are left to the converter warps.
      uint64_t pol_w;
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_w));
      Cursor W;
      bool more = W.next(a, c, G);
      RingPos rq;
      long long ir = 0;
      bool ok = true;
      while (more && ok) {
        const StackPhase& P = a.ph[W.p];
        if (P.w4) {
          const int j = rq.s;
          if (rq.r > 0 && !mbar_wait(&rempty[j], (rq.r - 1) & 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&rfull[j], (uint32_t)kInt4BlockBytes);
          bulk_load_hint(rraw + (size_t)j * kInt4BlockBytes,
                         P.w4 + ((size_t)W.sl * P.kbt + W.kb) * kInt4BlockBytes, (uint32_t)kInt4BlockBytes,
                         &rfull[j], pol_w);
          ++ir;
          rq.step(a.rw);
        }
        more = W.advance(a, c, G);
      }
      if (!ok) {
        for (long long j = (ir > a.rw ? ir - a.rw : 0); j < ir; ++j) {
          const unsigned long long t0 = globaltimer();
          while (!mbar_try_wait(&rfull[j % a.rw], (uint32_t)(j / a.rw) & 1) && globaltimer() - t0 < kTimeoutNs) {
          }
        }
      }
    }
  } else if (W4 && warp >= kConvWarp) {
    // ------------------------------------------------------------ converter warps (int4 variant)
    // The units are dealt round-robin over nc = min(4, S) warps: warp cw expands
    // units cw, cw + nc, ... (all 128 weight rows, four per lane) into the unit's
    // slot once the MMA has released it, so nc units are in conversion at once.
    // Row r's 16-byte chunk ch goes to chunk ch ^ (r & 7) of the row: the layout
    // TMA's 128-byte swizzle writes. A unit of a 16-bit phase gets its bf16 box by
    // TMA instead, issued by the same warp.
    // nc <= S keeps the parity waits exact: a warp waits for the release of unit
    // i - S only after its previous unit i - nc waited for unit i - nc - S, so the
    // slot's barrier is never two phases behind the one it tests (a parity test
    // against a barrier two phases behind would pass at once).
    const int cw = warp - kConvWarp;
    const int nc = S < 4 ? S : 4;
    uint64_t pol_w;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_w));
    Cursor K;
    bool more = K.next(a, c, G);
    RingPos sp, rq;   // slots (every unit), packed blocks (int4 units)
    long long iu = 0, nb = 0;  // units passed, bf16 boxes issued by this warp
    int cur_p = -1;
    const uint8_t* cur_w4 = nullptr;  // the current phase's packed weight (read once per phase)
    bool ok = cw < nc;
    while (more && ok) {
      if (K.p != cur_p) {
        cur_p = K.p;
        cur_w4 = a.ph[K.p].w4;
      }
      const int s = sp.s;
      if ((int)(iu % nc) == cw) {
        if (sp.r > 0) {
          bool w = true;
          if (lane == 0) w = mbar_wait(&empty[s], (sp.r - 1) & 1, abort_flag, a.status);
          if (!__shfl_sync(0xffffffffu, (int)w, 0)) {
            ok = false;
            break;
          }
        }
        if (cur_w4) {
          const int j = rq.s;
          bool w = true;
          if (lane == 0) w = mbar_wait(&rfull[j], rq.r & 1, abort_flag, a.status);
          if (!__shfl_sync(0xffffffffu, (int)w, 0)) {
            ok = false;
            break;
          }
          const uint8_t* raw = rraw + (size_t)j * kInt4BlockBytes;
          uint8_t* slot = wring + (size_t)s * wslot;
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            const int r = rr * 32 + lane;
            const uint4 q0 = *reinterpret_cast<const uint4*>(raw + r * 32);
            const uint4 q1 = *reinterpret_cast<const uint4*>(raw + r * 32 + 16);
            const __nv_bfloat16 sc = reinterpret_cast<const __nv_bfloat16*>(raw + kInt4CodeBytes)[r];
            const __nv_bfloat162 s2 = __halves2bfloat162(sc, sc);
            uint8_t* dst = slot + r * 128;
            const uint32_t wd[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(dst + ((ch ^ (r & 7)) << 4)) = int4_dequant8(wd[ch], s2);
          }
          // the MMA reads the slot through the async proxy
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&rempty[j]);
            mbar_arrive(&full[s]);
          }
        } else if (lane == 0) {  // a 16-bit phase: its bf16 box, as the plain variant's weight producer loads it
          mbar_expect_tx(&full[s], (uint32_t)kWBytes);
          tma_load_2d_hint(wring + (size_t)s * wslot, &a.ph[K.p].tmW, &full[s], K.kb * kBK, K.sl * kTileN, pol_w);
          ++nb;
        }
      }
      if (cur_w4) rq.step(a.rw);
      ++iu;
      sp.step(S);
      more = K.advance(a, c, G);
    }
    if (!ok && nb > 0 && lane == 0) {
      for (long long j = (iu > S ? iu - S : 0); j < iu; ++j) {
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(&full[j % S], (uint32_t)(j / S) & 1) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
    }
  } else if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ weight producer
      // Weight boxes depend on no phase: stream them through the ring as fast as
      // the MMA frees stages, across phase boundaries.
      uint64_t pol_w;  // weights are read once
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_w));
      // (Prefetching further weight boxes into L2 while the ring is full was
      // measured slower: the extra requests delay the ring's own loads and the
      // attention phase's KV reads.)
      Cursor W;
      bool more = W.next(a, c, G);
      RingPos rp;
      long long iw = 0;  // units loaded into the ring
      bool ok = true;
      while (more && ok) {
        const int s = rp.s;
        if (rp.r > 0 && !mbar_wait(&empty[s], (rp.r - 1) & 1, abort_flag, a.status)) {
          ok = false;
          break;
        }
        mbar_expect_tx(&full[s], (uint32_t)kWBytes);
        tma_load_2d_hint(wring + (size_t)s * wslot, &a.ph[W.p].tmW, &full[s], W.kb * kBK, W.sl * kTileN, pol_w);
        ++iw;
        rp.step(S);
        more = W.advance(a, c, G);
      }
      if (!ok) {
        // drain (bounded): every box issued must land before the CTA exits
        for (long long j = (iw > S ? iw - S : 0); j < iw; ++j) {
          const unsigned long long t0 = globaltimer();
          while (!mbar_try_wait(&full[j % S], (uint32_t)(j / S) & 1) && globaltimer() - t0 < kTimeoutNs) {
          }
        }
      }
    }
  } else if (warp == kXWarp) {
    if (lane == 0) {
      // ------------------------------------------------------------ activation producer
      // The activation boxes of phase p wait until every CTA has finished phase p - 1.
      uint64_t pol_x;  // activations are read by every CTA
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_x));
      Cursor X;
      bool more = X.next(a, c, G);
      RingPos rp;
      long long ix = 0;
      int ready = -1;
      bool ok = true;
      while (more && ok) {
        if (ready != X.p) {
          if (X.p > 0 && !wait_phase(a, X.p - 1, (unsigned)G, abort_flag)) {
            ok = false;
            break;
          }
          fence_proxy_async();  // the phase's activations were written by other CTAs' generic stores
          ready = X.p;
        }
        const int s = rp.s;
        if (rp.r > 0 && !mbar_wait(&empty[s], (rp.r - 1) & 1, abort_flag, a.status)) {
          ok = false;
          break;
        }
        const StackPhase& P = a.ph[X.p];
        uint8_t* dst = xring + (size_t)s * xbytes;
        mbar_expect_tx(&full[s], (uint32_t)xbytes);
        tma_load_2d_hint(dst, &P.tmX, &full[s], X.kb * kBK, 0, pol_x);
        if (a.has_lo) tma_load_2d_hint(dst + xbox, &P.tmXlo, &full[s], X.kb * kBK, 0, pol_x);
        ++ix;
        rp.step(S);
        more = X.advance(a, c, G);
      }
      if (!ok) {
        for (long long j = (ix > S ? ix - S : 0); j < ix; ++j) {
          const unsigned long long t0 = globaltimer();
          while (!mbar_try_wait(&full[j % S], (uint32_t)(j / S) & 1) && globaltimer() - t0 < kTimeoutNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      // hi/lo pairs: one MMA of N = 2 MT over both boxes (hi products in accumulator
      // columns [0, MT), lo ones in [MT, 2 MT), added by the epilogue)
      const uint32_t idesc = idesc_bf16(a.has_lo ? 2 * MT : MT);
      Cursor C;
      bool more = C.next(a, c, G);
      RingPos rp;
      int f = 0;
      bool ok = true;
      while (more && ok) {
        const int kb0 = C.kb, kb1 = min(C.kbt, kb0 + (C.u1 - C.u));  // this tile's k-blocks in the range
        const int buf = f & 1;
        if (f >= 2 && !mbar_wait(&aempty[buf], (uint32_t)((f >> 1) - 1) & 1, abort_flag, a.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * abufw);
        for (int kb = kb0; kb < kb1; ++kb) {
          const int sw = rp.s, sx = sw;
          if (!mbar_wait(&full[sw], rp.r & 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t aw = smem_u32(wring + (size_t)sw * wslot);
          const uint32_t ax = smem_u32(xring + (size_t)sx * xbytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            umma(d, sw128_desc(aw + k * 32), sw128_desc(ax + k * 32), idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          umma_commit(&empty[sw]);
          rp.step(S);
        }
        if (!ok) break;
        umma_commit(&afull[buf]);
        ++f;
        more = C.advance(a, c, G, kb1 - kb0);
      }
      // no MMA may still be writing tensor memory when it is freed
      umma_commit(drain);
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < kTimeoutNs) {
      }
    }
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------------------------ epilogue, attention, merge
    const int etid = threadIdx.x - 64;
    const int ew = etid >> 5;             // epilogue warp 0..3
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int col = q * 32 + lane;        // weight row within the tile = output column
    const int rows_valid = min(MT, a.M);
    int f = 0;
    bool alive = true;
    attn::UmState ust;  // attention items: staging at the activation ring, S / O in TMEM columns [0, 256)
    ust.groups = sgroups;
    ust.sm = xring;
    ust.kv_bar = at_kv;
    ust.mma_bar = at_mma;
    ust.tmem = tmem;
    // The attention phases of a program share their rows and groups: this CTA's
    // items and merge pairs are decoded once, while the first phase streams.
    struct {
      int n0 = 1, slots = 0, i0 = 0, i1 = 0, w0 = 0, w1 = 0;
      attn::UmItem first{};
    } plan;
    if (a.first_attn >= 0) {
      const AttnArgs& at = a.ph[a.first_attn].at;
      const attn::UmItems items(at, sgroups, G);
      const int n = items.count(), nm = at.M * at.Hq;
      plan.n0 = items.n0;
      plan.slots = attn::um_part_slots(at.max_prefix, at.Hkv, kMaxCtas);
      plan.i0 = (int)((long long)c * n / G);
      plan.i1 = (int)((long long)(c + 1) * n / G);
      plan.w0 = (int)((long long)c * nm / G);
      plan.w1 = (int)((long long)(c + 1) * nm / G);
      if (plan.i0 < plan.i1) items.item(plan.i0, plan.first.chunk, plan.first.kvh, plan.first.rt, plan.first.z);
    }
    for (int p = 0; p < a.n_phases; ++p) {
      const StackPhase& P = a.ph[p];
      if (p > 0 && alive) alive = epi_all(etid != 0 || wait_phase(a, p - 1, (unsigned)G, abort_flag));
      if (alive && P.kind == kPhaseGemm) {
        EpiParams ep = P.ep;
        if (a.y_last && p == a.n_phases - 1) ep.y = a.y_last;
        // the phase's row inputs (RMSNorm scales, RoPE rows) once, while the first
        // accumulator streams in
        load_epi_rows(ep, 0, rows_valid, prow, etid, kEpiThreads);
        EpilogueSync{}();
        const int kbt = P.kbt;
        const Split sp(P, G);
        int ua0, ua1, ub0, ub1;
        sp.split_range(c, ua0, ua1);
        sp.whole_range(c, ub0, ub1);
        const int t_first = ua0 < ua1 ? (int)(ua0 / kbt) : 0;
        int seg_t[2], nseg = 0;  // split tiles of this CTA in this phase (its first and last at most)
        // the split range, then (after the fixup below) the whole tiles
        auto run_units = [&](int u0, int u1) {
        for (int u = u0; u < u1 && alive;) {
          const int t = u / kbt;
          const int kb0 = u - t * kbt;
          const int kb1 = min(kbt, u1 - t * kbt);
          const bool whole = kb0 == 0 && kb1 == kbt;
          const int buf = f & 1;
          const bool ok = epi_all(mbar_wait(&afull[buf], (uint32_t)(f >> 1) & 1, abort_flag, a.status));
          tc_fence_after();
          const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * abufw);
          if (!ok) {
            alive = false;
          } else if (whole) {
            const int n0 = t * kTileN;
            for (int r0 = 0; r0 < rows_valid; r0 += kSub) {
              float v[32];
              tmem_ld32_pair(tb + r0, a.has_lo ? MT : 0, v);
#pragma unroll
              for (int i = 0; i < 32; ++i) tile[i * kLdt + col] = v[i];
              EpilogueSync{}();
              epilogue_body<bf16>(ep, tile, kLdt, r0, min(kSub, rows_valid - r0), n0, prow.at(r0), etid,
                                 EpilogueSync{});
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&aempty[buf]);
          } else {
            // split tile: leave the fragment in this CTA's slot and count it in; the
            // tile is finished after the split range, once every fragment is in
            float* slot = a.partial + ((size_t)c * 2 + (t != t_first ? 1 : 0)) * (size_t)MT * kTileN;
            for (int r0 = 0; r0 < rows_valid; r0 += kSub) {
              float v[32];
              tmem_ld32_pair(tb + r0, a.has_lo ? MT : 0, v);
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (r0 + i < rows_valid) __stcg(slot + (size_t)(r0 + i) * kTileN + col, v[i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&aempty[buf]);
            EpilogueSync{}();
            if (etid == 0) {  // the barrier orders the other threads' stores before this fence
              __threadfence();
              red_release_add(reinterpret_cast<unsigned*>(a.tile_cnt + P.cnt_off + t), 1u);
            }
            seg_t[nseg++] = t;
          }
          ++f;
          u = (t + 1) * kbt;
        }
        };
        run_units(ua0, ua1);
        // Distributed fixup: the n CTAs that share a split tile each sum one slice
        // of its rows over all n fragments, in ascending CTA order (the standalone
        // GEMM's order), and run the epilogue on that slice. Every CTA of the
        // cooperative launch is resident, so waiting for the others' fragments is safe.
        for (int si = 0; si < nseg && alive; ++si) {
          const int t = seg_t[si];
          int c0, c1;
          sp.sharers(t, c0, c1);
          const int nc = c1 - c0 + 1, me = c - c0;
          // fragment slot: CTAs after c0 start their split range inside tile t (slot 0);
          // c0 holds t in slot 1 when its range starts in an earlier tile
          const int slot_c0 = sp.first_split_tile(c0) != t ? 1 : 0;
          const int r_lo = me * rows_valid / nc, r_hi = (me + 1) * rows_valid / nc;
          alive = epi_all(etid != 0 || wait_count(a, P.cnt_off + t, (unsigned)nc, abort_flag));
          if (!alive || r_lo >= r_hi) continue;
          const int n0 = t * kTileN;
          for (int rb0 = r_lo; rb0 < r_hi; rb0 += kSub) {
            const int nr = min(kSub, r_hi - rb0);
            const int pairs = nr * (kTileN / 4);  // (row, 4-column group) pairs of this block
            for (int p0 = 0; p0 < pairs; p0 += 4 * kEpiThreads) {
              float4 acc[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int cb = c0; cb <= c1; cb += 4) {
                // up to 4 fragments x 4 pairs of loads in flight, added in CTA order
                float4 x[4][4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const int cc = cb + k;
                  const float* fp =
                      cc <= c1 ? a.partial + ((size_t)cc * 2 + (cc == c0 ? slot_c0 : 0)) * (size_t)MT * kTileN
                               : nullptr;
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    const int pr = p0 + i * kEpiThreads + etid;
                    x[k][i] = (fp && pr < pairs)
                                  ? __ldcg(reinterpret_cast<const float4*>(fp + (size_t)(rb0 + pr / 32) * kTileN +
                                                                           (pr % 32) * 4))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                  }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  if (cb + k > c1) break;
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    acc[i].x += x[k][i].x; acc[i].y += x[k][i].y; acc[i].z += x[k][i].z; acc[i].w += x[k][i].w;
                  }
                }
              }
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int pr = p0 + i * kEpiThreads + etid;
                if (pr < pairs) {
                  float* tr = tile + (pr / 32) * kLdt + (pr % 32) * 4;
                  tr[0] = acc[i].x; tr[1] = acc[i].y; tr[2] = acc[i].z; tr[3] = acc[i].w;
                }
              }
            }
            EpilogueSync{}();
            epilogue_body<bf16>(ep, tile, kLdt, rb0, nr, n0, prow.at(rb0), etid, EpilogueSync{});
          }
        }
        run_units(ub0, ub1);
      } else if (alive && P.kind == kPhaseAttn) {
        const AttnArgs& at = P.at;
        attn::UmItem cur = plan.first, nxt{};
        if (plan.i0 < plan.i1) {
          // the tiles alias the activation ring and the epilogue tile: fence this
          // thread's generic writes there before the copies overwrite them
          attn::fence_proxy_async_smem();
          EpilogueSync{}();
          if (etid == 0) attn::um_issue<HD>(at, &P.tmXlo, &P.tmW, &P.tmX, cur, plan.n0, ust);
        }
        for (int i = plan.i0; i < plan.i1 && alive; ++i) {
          const bool has_next = i + 1 < plan.i1;
          if (has_next) attn::UmItems(at, sgroups, G).item(i + 1, nxt.chunk, nxt.kvh, nxt.rt, nxt.z);
          alive = attn::attn_item_um<HD>(at, &P.tmXlo, &P.tmW, &P.tmX, cur, has_next, nxt, plan.n0, plan.slots, ust,
                                         etid, col, abort_flag, EpilogueSync{});
          cur = nxt;
        }
      } else if (alive && P.kind == kPhaseMerge) {
        // the attention items' staging region is free (their phase is complete)
        alive = attn::um_merge_staged<HD>(P.at, sgroups, plan.n0, plan.w0, plan.w1, plan.slots, xring,
                                          (uint32_t)attn::um_smem_bytes<HD>(), at_kv, &ust.kv_par, etid,
                                          abort_flag, EpilogueSync{});
      }
      // phase done: every epilogue thread's writes happen before the release
      EpilogueSync{}();
      if (etid == 0) {
        __threadfence();
        fence_proxy_async();
        red_release_add(a.done + p, 1u);
        if (a.trace) a.trace[(size_t)p * G + c] = globaltimer();
      }
    }
    // The LM head's top-k records merged in the same launch (instead of a kernel
    // of its own after it): once every CTA has finished the last phase, CTA c
    // merges row c (M <= 128 rows, fewer than CTAs) with its epilogue threads.
    if (alive && a.mg.k > 0 && c < a.mg.M) {
      alive = epi_all(etid != 0 || wait_phase(a, a.n_phases - 1, (unsigned)G, abort_flag));
      if (alive) topk_merge_row<kEpiThreads>(a.mg, c, etid, tile, EpilogueSync{});
    }
  }
  // the producer and MMA roles ran on lane 0 only: reconverge each warp before the
  // block barrier and the warp-wide (.sync.aligned) TMEM dealloc
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    // the last CTA out returns every counter to zero for the next launch
    __threadfence();
    const unsigned prev = atomicAdd(a.done + a.n_phases, 1u);
    *exit_last = prev == (unsigned)(G - 1);
  }
  __syncthreads();
  if (*exit_last) {
    __threadfence();
    for (int i = threadIdx.x; i <= a.n_phases; i += NT) a.done[i] = 0u;
    for (int i = threadIdx.x; i < a.n_counters; i += NT) a.tile_cnt[i] = 0;
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols) : "memory");
  }
}

struct Layout {
  int sw, sx, apad, rw;
  size_t smem;
};

// Ring stages: as many as fit once the attention tiles (aliasing the activation
// halves and the epilogue tile, padded where those are smaller) are accounted for.
Layout layout(int MT, bool has_lo, int hd, bool w4) {
  Layout l{};
  const size_t xbytes = (size_t)MT * kBK * 2 * (has_lo ? 2 : 1);
  const size_t wslot = kWBytes;
  const size_t attn = hd == 128 ? attn::um_smem_bytes<128>() : attn::um_smem_bytes<64>();
  const size_t fixed = kTileBytes + (size_t)(2 * kMaxW + 7) * 8 + 16 + kMaxGroups * sizeof(Group) + 1024;
  if (w4) {
    // int4 variant: as many slots (up to 6) as leave room for at least 10
    // packed-block stages (4352 bytes + two barriers each; else 4), then as many
    // stages as fit. At least as many stages as slots: a converter tests a stage's
    // barrier only after the unit R stages back was consumed, which keeps that
    // parity test exact too.
    for (int pass = 0; pass < 2; ++pass)
    for (int s = 6; s >= 2; --s) {
      const size_t alias = (size_t)s * xbytes + kTileBytes;
      const size_t pad = alias >= attn ? 0 : (attn - alias + 15) / 16 * 16;
      const size_t smem = (size_t)s * (wslot + xbytes) + fixed + pad + 16;
      if (smem >= (size_t)kSmemBudget) continue;
      const int r = (int)std::min<size_t>(kMaxRaw, ((size_t)kSmemBudget - smem) / (kInt4BlockBytes + 16));
      if (r < std::max(s, pass == 0 ? 10 : 4)) continue;
      l.sw = l.sx = s;
      l.rw = r;
      l.apad = (int)pad;
      l.smem = smem + (size_t)r * (kInt4BlockBytes + 16);
      return l;
    }
    return l;
  }
  for (int s = kMaxW; s >= 2; --s) {
    const size_t alias = (size_t)s * xbytes + kTileBytes;
    const size_t pad = alias >= attn ? 0 : (attn - alias + 15) / 16 * 16;
    const size_t smem = (size_t)s * (wslot + xbytes) + fixed + pad;
    if (smem <= (size_t)kSmemBudget) {
      l.sw = l.sx = s;
      l.apad = (int)pad;
      l.smem = smem;
      return l;
    }
  }
  return l;  // sw = 0: rejected by stack_run
}

int round_mt(int M) {
  int MT = ((M + 31) / 32) * 32;
  return MT < 32 ? 32 : MT;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace

int stack_mt(int M) { return round_mt(M); }

int stack_ctas() { return num_sms(); }

bool stack_supported(int M, int hd) { return M >= 1 && M <= kStackMaxRows && (hd == 64 || hd == 128); }

size_t stack_scratch_bytes(int M, int max_phases, int max_counters) {
  return align256((size_t)(max_phases + 1) * 4) + align256((size_t)max_counters * 4) +
         (size_t)kMaxCtas * 2 * round_mt(M) * kTileN * 4;  // [CTA][first/last split tile][rows][128]
}

size_t stack_attention_part_bytes(int M, int Hq, int Hkv, int hd, int max_prefix) {
  const size_t slots = (size_t)attn::um_part_slots(max_prefix, Hkv, kMaxCtas);
  return (size_t)M * Hq * slots * (hd + 2) * sizeof(float);
}

void StackProgramBuilder::gemm(const StackGemmDesc& g) {
  StackPhase ph{};
  ph.kind = kPhaseGemm;
  ph.N = g.N;
  ph.K = g.K;
  if (g.N % kTileN || g.K % kBK || g.rows_cap < M || !g.W || !g.X) { ok = false; return; }
  if (((reinterpret_cast<uintptr_t>(g.W) | reinterpret_cast<uintptr_t>(g.X) |
        reinterpret_cast<uintptr_t>(g.X_lo)) & 15) != 0) { ok = false; return; }
  if (has_lo != (g.X_lo != nullptr)) { ok = false; return; }
  ph.n_tiles = g.N / kTileN;
  ph.kbt = g.K / kBK;
  // (Two-tile units sharing one activation box were measured slower: more
  // sharers per split tile and a shallower ring.)
  ph.T = (long long)ph.n_tiles * ph.kbt;
  ph.cnt_off = n_counters;
  n_counters += ph.n_tiles;  // one arrival counter per tile
  ph.ep = g.ep;
  ph.ep.M = M;
  if (g.w4) {
    ph.w4 = reinterpret_cast<const uint8_t*>(g.W);  // blocks of 128 x 64, 16-byte aligned (checked above)
    has_w4 = true;
  }
  if ((!g.w4 && !make_tmap_bf16(&ph.tmW, g.W, g.N, g.K, kTileN)) ||
      !make_tmap_bf16(&ph.tmX, g.X, g.rows_cap, g.K, MT) ||
      (g.X_lo && !make_tmap_bf16(&ph.tmXlo, g.X_lo, g.rows_cap, g.K, MT))) {
    ok = false;
    return;
  }
  if (!g.X_lo) ph.tmXlo = ph.tmX;
  phases.push_back(ph);
}

void StackProgramBuilder::attention(const AttnArgs& a) {
  StackPhase ph{};
  ph.kind = kPhaseAttn;
  ph.at = a;
  ph.at.M = M;
  // the items copy 128 rows (keys, or GQA query rows) x 64 halves per box
  const long long rows = (long long)a.n_seq * a.Hkv * a.cap;
  const long long qrows = (long long)M * a.Hq;  // [Hkv][M][Hq / Hkv] query rows
  if (rows <= 0 || rows > (1ll << 31) - 1 || (a.hd != 64 && a.hd != 128) || !a.qg ||
      !make_tmap_f16(&ph.tmW, a.kc, (int)rows, a.hd, attn::kUmKeys) ||
      !make_tmap_f16(&ph.tmX, a.vc, (int)rows, a.hd, attn::kUmKeys) ||
      !make_tmap_f16(&ph.tmXlo, a.qg, (int)qrows, a.hd, attn::kUmRows)) {
    ok = false;
    return;
  }
  if (first_attn < 0) first_attn = (int)phases.size();
  phases.push_back(ph);
  ph.kind = kPhaseMerge;
  phases.push_back(ph);
}

cudaError_t stack_run(const StackPhase* d_phases, int n_phases, int M, bool has_lo, int hd, int n_counters,
                      void* scratch, int max_phases, int max_counters, int* status, unsigned long long* trace,
                      float* y_last, const Group* groups, int n_groups, int first_attn, cudaStream_t s,
                      bool w4, const TopkMerge* merge) {
  if (!stack_supported(M, hd) || n_phases <= 0 || !scratch || n_phases > max_phases || n_counters > max_counters)
    return cudaErrorInvalidValue;
  if (n_groups < 0 || n_groups > kMaxGroups || (n_groups > 0 && !groups)) return cudaErrorInvalidValue;
  const int MT = round_mt(M);
  const Layout l = layout(MT, has_lo, hd, w4);
  if (l.sw < 2) return cudaErrorInvalidValue;
  StackArgs a{};
  a.ph = d_phases;
  a.n_phases = n_phases;
  a.M = M;
  a.MT = MT;
  a.has_lo = has_lo;
  a.sw = l.sw;
  a.sx = l.sx;
  a.rw = l.rw;
  a.apad = l.apad;
  uint32_t cols = attn::kUmTmemCols;  // attention S and O
  while (cols < (uint32_t)(2 * (has_lo ? 2 * MT : MT))) cols <<= 1;  // two accumulator buffers
  a.tmem_cols = cols;
  // the layout depends only on the capacities, never on this program: programs
  // of every size share one scratch
  char* base = reinterpret_cast<char*>(scratch);
  a.done = reinterpret_cast<unsigned*>(base);
  base += align256((size_t)(max_phases + 1) * 4);
  a.tile_cnt = reinterpret_cast<int*>(base);
  a.n_counters = n_counters;
  base += align256((size_t)max_counters * 4);
  a.partial = reinterpret_cast<float*>(base);
  a.status = status;
  a.trace = trace;
  a.y_last = y_last;
  a.groups = groups;
  a.n_groups = n_groups;
  a.first_attn = first_attn < n_phases ? first_attn : -1;
  if (merge && merge->k > 0) {
    if (merge->k > kMaxTopK || merge->M > M || merge->M > num_sms() || !merge->out_idx || !merge->val ||
        !merge->idx || !merge->mx || !merge->sum || merge->ntiles < 1)
      return cudaErrorInvalidValue;
    a.mg = *merge;
  }
  auto kernel = w4 ? (hd == 128 ? stack_tc_kernel<128, true> : stack_tc_kernel<64, true>)
                   : (hd == 128 ? stack_tc_kernel<128, false> : stack_tc_kernel<64, false>);
  if (!raise_smem_limit(reinterpret_cast<const void*>(kernel), kSmemBudget)) return cudaErrorInvalidValue;
  const int G = num_sms();
  if (G > kMaxCtas) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(w4 ? kThreadsW4 : kThreads);
  cfg.dynamicSmemBytes = l.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident at once: phases wait on each other
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace eg

// ------------------------------------------------------------------ op entry point
namespace eg {
namespace {
size_t op_prog_bytes(int n_phases) { return align256((size_t)n_phases * sizeof(StackPhase)); }
size_t op_rec_bytes(int M, int N, int k) {
  const size_t nt = (size_t)((N + kTileN - 1) / kTileN) * M;
  return k > 0 ? 2 * align256(nt * k * 4) + 2 * align256(nt * 4) : 0;
}
}  // namespace
}  // namespace eg

extern "C" {

size_t eagle_op_gemm_persistent_scratch_bytes(int32_t M, int32_t N, int32_t K, int32_t n_phases, int32_t k) {
  using namespace eg;
  if (M < 1 || N < 1 || K < 1 || n_phases < 1 || k < 0 || k > kMaxTopK) return 0;
  return op_prog_bytes(n_phases) + op_rec_bytes(M, N, k) +
         stack_scratch_bytes(M, n_phases, n_phases * ((N + kTileN - 1) / kTileN));
}

eagle_status eagle_op_gemm_persistent(int32_t M, int32_t N, int32_t K, int32_t n_phases, int32_t k, const void* x,
                                      const void* x_lo, const void* w, float* y, int32_t* idx, float* val,
                                      float* lse, void* scratch, size_t scratch_bytes, void* stream) {
  using namespace eg;
  if (M < 1 || N < 1 || K < 1 || n_phases < 1 || k < 0 || k > kMaxTopK || !x || !w || !scratch)
    return EAGLE_ERR_INVALID_ARG;
  if ((k == 0 || n_phases > 1) && !y) return EAGLE_ERR_INVALID_ARG;
  if (k > 0 && !idx) return EAGLE_ERR_INVALID_ARG;
  if (!stack_supported(M, 128) || N % kTileN || K % kBK) return EAGLE_ERR_UNSUPPORTED;
  if (scratch_bytes < eagle_op_gemm_persistent_scratch_bytes(M, N, K, n_phases, k)) return EAGLE_ERR_WORKSPACE;
  char* p = reinterpret_cast<char*>(scratch);
  StackPhase* d_prog = reinterpret_cast<StackPhase*>(p);
  p += op_prog_bytes(n_phases);
  const size_t nt = (size_t)((N + kTileN - 1) / kTileN) * M;
  EpiParams lm;
  lm.kind = kEpiLmHead;
  lm.N = N;
  lm.topk = k;
  if (k > 0) {
    lm.rec_val = reinterpret_cast<float*>(p); p += align256(nt * k * 4);
    lm.rec_idx = reinterpret_cast<int*>(p); p += align256(nt * k * 4);
    lm.rec_max = reinterpret_cast<float*>(p); p += align256(nt * 4);
    lm.rec_sum = reinterpret_cast<float*>(p); p += align256(nt * 4);
  }
  StackProgramBuilder b;
  b.M = M;
  b.MT = stack_mt(M);
  b.has_lo = x_lo != nullptr;
  EpiParams st;
  st.kind = kEpiStore;
  st.N = N;
  st.y = y;
  for (int i = 0; i < n_phases; ++i)
    b.gemm(StackGemmDesc{(const bf16*)w, (const bf16*)x, (const bf16*)x_lo, M, N, K,
                         (k > 0 && i == n_phases - 1) ? lm : st});
  if (!b.ok) return EAGLE_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(d_prog, b.phases.data(), b.phases.size() * sizeof(StackPhase), cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return EAGLE_ERR_CUDA;
  TopkMerge mg;  // the top-k merge runs inside the launch, after the LM-head phase
  if (k > 0) {
    mg.val = lm.rec_val;
    mg.idx = lm.rec_idx;
    mg.mx = lm.rec_max;
    mg.sum = lm.rec_sum;
    mg.ntiles = (N + kTileN - 1) / kTileN;
    mg.M = M;
    mg.k = k;
    mg.out_idx = idx;
    mg.out_val = val;
    mg.out_lse = lse;
  }
  cudaError_t err = stack_run(d_prog, n_phases, M, x_lo != nullptr, 128, b.n_counters, p, n_phases, b.n_counters,
                              nullptr, nullptr, nullptr, nullptr, 0, -1, s, false, &mg);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);  // b.phases is a host temporary
  return err == cudaSuccess ? EAGLE_OK : (err == cudaErrorInvalidValue ? EAGLE_ERR_UNSUPPORTED : EAGLE_ERR_CUDA);
}

}  // extern "C"
