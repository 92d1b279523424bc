// Weight-streaming GEMM Y = X W^T on the sm_103a tensor cores (tcgen05 + TMA).
//
// The verify pass multiplies a few dozen token rows by every weight matrix of
// the target, so it is bound by streaming the weights from HBM. Swap-AB: a
// 128-row weight tile is the UMMA M operand (A, K-major, 128B-swizzled, loaded
// by TMA), the token rows are the UMMA N operand (B, N = 32..256), and the
// fp32 accumulator lives in tensor memory. The (tile, 64-wide k-block) units of
// a GEMM are split evenly over the SMs (stream-K); a tile cut between CTAs is
// summed by the CTA that finishes it last, over the CTAs in ascending order,
// so every output is summed in an order that depends only on (N, K) and the SM
// count, never on M or on timing.
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0     TMA producer (one lane): W box [128 x 64] + X box [MT x 64] per stage
//   warp 1     TMEM allocator and MMA issuer (one lane): 4 x tcgen05.mma (K = 16) per stage
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//              32 (w % 4) ..), fixup, then the shared epilogue on 32-row sub-tiles
// Every mbarrier wait is bounded (2 s of %globaltimer); a timeout sets the
// device status word and an abort flag that the other roles observe, and the
// kernel drains and frees its tensor memory before returning.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <utility>
#include <vector>

#include "../../include/eagle.h"
#include "epilogue.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace eg {
namespace {

constexpr int kThreads = 192;
constexpr int kBK = 64;                       // K elements per stage: one 128-byte swizzle row
constexpr int kWBytes = kTileN * kBK * 2;     // 16 KB weight box
constexpr int kSub = 32;                      // epilogue rows per sub-tile
constexpr int kLdt = kTileN + 1;
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 232448;           // 227 KB opt-in per block
constexpr int kNsmSizing = 160;               // SM count bound used for scratch sizing
// Split-K arrival counters sit at the start of the scratch in a region of fixed
// size, so that one scratch buffer serves GEMMs of every shape: a shape's
// partial sums can never land on another shape's counters.
constexpr int kCounterInts = 1 << 17;
constexpr size_t kCounterBytes = (size_t)kCounterInts * 4;
// Allocation-free variant (eagle_op_gemm_noalloc): token rows <= 64, so the
// partial sums need at most kNsmSizing CTAs x 2 fragments x 64 rows x 128 columns.
constexpr int kNoAllocMaxM = 64;
constexpr size_t kNoAllocScratchBytes = kCounterBytes + (size_t)kNsmSizing * 2 * 64 * kTileN * 4;

struct TcArgs {
  int M, MT, m_chunks, n_tiles, kbt, G, stages;
  int has_lo;      // activations come as a hi/lo pair: a second X box per stage, right after the first
  int wide;        // has_lo and 2 MT <= 256: one MMA of N = 2 MT per k-step covers both boxes, the
                   // accumulator holds the hi products in columns [0, MT) and the lo ones in [MT, 2 MT)
  long long T;
  uint32_t tmem_cols;
  int w_dep;       // the weights were written by the previous kernel: wait for it before loading them
  int* counters;   // [m_chunks][n_tiles], zero on entry and on exit
  float* partial;  // [m_chunks][G][2][MT][128]
  int* status;
};

using namespace tc;

// ------------------------------------------------------------------ schedule
__device__ __forceinline__ long long unit_start(const TcArgs& a, int c) { return (long long)c * a.T / a.G; }
__device__ __forceinline__ int cta_of(const TcArgs& a, long long u) {
  return (int)(((u + 1) * a.G - 1) / a.T);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmXlo, TcArgs a, EpiParams ep) {
  extern __shared__ uint8_t smem_raw[];
  // an offset from the shared array keeps the pointers in the shared address space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int S = a.stages, MT = a.MT;
  const int xbytes = MT * kBK * 2;
  const int stage_bytes = kWBytes + xbytes * (a.has_lo ? 2 : 1);
  uint8_t* stage_base = smem;
  float* tile = reinterpret_cast<float*>(smem + (size_t)S * stage_bytes);
  float* rscale = tile + kSub * kLdt;
  uint64_t* bars = reinterpret_cast<uint64_t*>(rscale + kEpiRowSmemFloats);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* afull = bars + 2 * S;
  uint64_t* aempty = bars + 2 * S + 2;
  uint64_t* drain = bars + 2 * S + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x / a.m_chunks, mc = blockIdx.x % a.m_chunks;
  const int m0 = mc * MT;
  const long long u0 = unit_start(a, c), u1 = unit_start(a, c + 1);
  const int kbt = a.kbt;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&afull[b], 1);
      mbar_init(&aempty[b], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    *last_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
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
  if (threadIdx.x == 0) griddep_launch();  // the next kernel may start its own prologue on freed SMs

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- TMA producer
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
      if (a.has_lo) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmXlo)) : "memory");
      uint64_t pol_w, pol_x;  // weights are read once per GEMM; activations by every CTA
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol_w));
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_x));
      // The weights do not depend on earlier kernels: request the weight boxes
      // of the first S stages before waiting for the previous kernel
      // (programmatic dependent launch), the activation boxes after it.
      int pre_kb[kMaxStages];
      int npre = 0;
      if (a.w_dep) griddep_wait();
      for (long long u = u0; u < u1 && npre < S; ++u, ++npre) {
        const int t = (int)(u / kbt);
        const int kb = (int)(u - (long long)t * kbt);
        mbar_expect_tx(&full[npre], (uint32_t)stage_bytes);
        tma_load_2d_hint(stage_base + (size_t)npre * stage_bytes, &tmW, &full[npre], kb * kBK, t * kTileN, pol_w);
        pre_kb[npre] = kb;
      }
      griddep_wait();
      for (int i = 0; i < npre; ++i) {
        uint8_t* sx = stage_base + (size_t)i * stage_bytes + kWBytes;
        tma_load_2d_hint(sx, &tmX, &full[i], pre_kb[i] * kBK, m0, pol_x);
        if (a.has_lo) tma_load_2d_hint(sx + xbytes, &tmXlo, &full[i], pre_kb[i] * kBK, m0, pol_x);
      }
      int it = npre;
      bool ok = true;
      for (long long u = u0 + npre; u < u1 && ok;) {
        const int t = (int)(u / kbt);
        const int kb0 = (int)(u - (long long)t * kbt);
        const int kb1 = (int)min((long long)kbt, u1 - (long long)t * kbt);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % S;
          if (it >= S && !mbar_wait(&empty[s], ((it / S) - 1) & 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          uint8_t* sw = stage_base + (size_t)s * stage_bytes;
          mbar_expect_tx(&full[s], (uint32_t)stage_bytes);
          tma_load_2d_hint(sw, &tmW, &full[s], kb * kBK, t * kTileN, pol_w);
          tma_load_2d_hint(sw + kWBytes, &tmX, &full[s], kb * kBK, m0, pol_x);
          if (a.has_lo) tma_load_2d_hint(sw + kWBytes + xbytes, &tmXlo, &full[s], kb * kBK, m0, pol_x);
        }
        u = (long long)(t + 1) * kbt;
      }
      if (!ok) {
        // drain: wait (bounded) for every load still in flight before the CTA exits
        for (int j = max(0, it - S); j < it; ++j) {
          const int s = j % S;
          const unsigned long long t0 = globaltimer();
          while (!mbar_try_wait(&full[s], (j / S) & 1) && globaltimer() - t0 < kTimeoutNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      const uint32_t idesc = idesc_bf16(a.wide ? 2 * MT : MT);
      const int accw = a.wide ? 2 * MT : MT;
      int it = 0, f = 0;
      bool ok = true;
      for (long long u = u0; u < u1 && ok;) {
        const int t = (int)(u / kbt);
        const int kb0 = (int)(u - (long long)t * kbt);
        const int kb1 = (int)min((long long)kbt, u1 - (long long)t * kbt);
        const int buf = f & 1;
        if (f >= 2 && !mbar_wait(&aempty[buf], ((f >> 1) - 1) & 1, abort_flag, a.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * accw);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % S;
          if (!mbar_wait(&full[s], (it / S) & 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sw = smem_u32(stage_base + (size_t)s * stage_bytes);
          const uint32_t sx = sw + kWBytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            umma(d, sw128_desc(sw + k * 32), sw128_desc(sx + k * 32), idesc, (kb > kb0 || k > 0) ? 1u : 0u);
            if (a.has_lo && !a.wide) umma(d, sw128_desc(sw + k * 32), sw128_desc(sx + xbytes + k * 32), idesc, 1u);
          }
          umma_commit(&empty[s]);
        }
        umma_commit(&afull[buf]);
        ++f;
        u = (long long)(t + 1) * kbt;
      }
      // no MMA may still be writing tensor memory when it is freed
      umma_commit(drain);
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(drain, 0) && globaltimer() - t0 < kTimeoutNs) {
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (128 threads)
    griddep_wait();                       // epilogue inputs (h, norms, rows) come from earlier kernels
    const int etid = threadIdx.x - 64;
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int col = q * 32 + lane;        // weight row within the tile = output column
    const int rows_valid = min(MT, a.M - m0);
    const int t_first = (int)(u0 / kbt);
    int f = 0;
    for (long long u = u0; u < u1;) {
      const int t = (int)(u / kbt);
      const int kb0 = (int)(u - (long long)t * kbt);
      const int kb1 = (int)min((long long)kbt, u1 - (long long)t * kbt);
      const bool whole = kb0 == 0 && kb1 == kbt;
      const int buf = f & 1;
      const bool ok = epi_all(mbar_wait(&afull[buf], (f >> 1) & 1, abort_flag, a.status));
      tc_fence_after();
      const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * (a.wide ? 2 * MT : MT));
      const int n0 = t * kTileN;
      if (whole) {
        for (int r0 = 0; r0 < rows_valid; r0 += kSub) {
          float v[32];
          tmem_ld32_pair(tb + r0, a.wide ? MT : 0, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) tile[j * kLdt + col] = ok ? v[j] : 0.f;
          EpilogueSync{}();
          if (ok) run_epilogue<bf16>(ep, tile, kLdt, m0 + r0, min(kSub, rows_valid - r0), n0, rscale, etid,
                                     EpilogueSync{});
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&aempty[buf]);
      } else {
        float* slot = a.partial + (((size_t)mc * a.G + c) * 2 + (t != t_first ? 1 : 0)) * (size_t)MT * kTileN;
        for (int r0 = 0; r0 < rows_valid; r0 += kSub) {
          float v[32];
          tmem_ld32_pair(tb + r0, a.wide ? MT : 0, v);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (r0 + j < rows_valid) slot[(size_t)(r0 + j) * kTileN + col] = v[j];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&aempty[buf]);
        __threadfence();
        EpilogueSync{}();
        const long long tu0 = (long long)t * kbt, tu1 = (long long)(t + 1) * kbt - 1;
        const int c0 = cta_of(a, tu0), c1 = cta_of(a, tu1);
        if (etid == 0) {
          int* cnt = a.counters + (size_t)mc * a.n_tiles + t;
          const int prev = atomicAdd(cnt, 1);
          const int last = prev == (c1 - c0);
          if (last) *cnt = 0;
          *last_flag = last;
        }
        EpilogueSync{}();
        if (*last_flag && ok) {
          __threadfence();
          for (int r0 = 0; r0 < rows_valid; r0 += kSub) {
            // fragments in ascending CTA order; the 32 rows of a fragment are loaded together
            float acc[kSub];
#pragma unroll
            for (int j = 0; j < kSub; ++j) acc[j] = 0.f;
            for (int cc = c0; cc <= c1; ++cc) {
              const int tf = (int)(unit_start(a, cc) / kbt);
              const float* sl = a.partial + (((size_t)mc * a.G + cc) * 2 + (t != tf ? 1 : 0)) * (size_t)MT * kTileN +
                                (size_t)r0 * kTileN + col;
              float v[kSub];
#pragma unroll
              for (int j = 0; j < kSub; ++j) v[j] = (r0 + j < rows_valid) ? __ldcg(sl + (size_t)j * kTileN) : 0.f;
#pragma unroll
              for (int j = 0; j < kSub; ++j) acc[j] += v[j];
            }
#pragma unroll
            for (int j = 0; j < kSub; ++j) tile[j * kLdt + col] = acc[j];
            EpilogueSync{}();
            run_epilogue<bf16>(ep, tile, kLdt, m0 + r0, min(kSub, rows_valid - r0), n0, rscale, etid,
                               EpilogueSync{});
          }
        }
      }
      ++f;
      u = (long long)(t + 1) * kbt;
    }
  }
  // warps 0 and 1 ran their role on lane 0 only: reconverge each warp before the
  // block barrier and the warp-wide (.sync.aligned) TMEM dealloc
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols) : "memory");
  }
}

// Failure-detection self-test: one thread waits, with the GEMM pipeline's
// bounded wait, on an mbarrier that nothing ever arrives on. The wait must give
// up after its time limit and report kStTimeout through the status word; the
// kernel then returns normally, so the context stays usable.
__global__ void bounded_wait_selftest_kernel(int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  abort_flag = 0;
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (mbar_wait(&bar, 0, &abort_flag, status)) set_status(status, 1);  // would mean the wait saw a phase flip
}

// ------------------------------------------------------------------ host side
}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_tmap_bf16(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_f16(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  // per device ordinal: a process may drive GPUs of different SM counts
  static int n_of[256] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) dev = 0;
  int n = n_of[dev];
  if (!n) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
    if (n > kNsmSizing) n = kNsmSizing;
    n_of[dev] = n;
  }
  return n;
}

bool raise_smem_limit(const void* kernel, int bytes) {
  // cudaFuncSetAttribute applies to the current device only: once per (kernel, device)
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& kd : done)
    if (kd.first == kernel && kd.second == dev) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  done.emplace_back(kernel, dev);
  return true;
}

namespace {

struct Plan {
  int MT, m_chunks, n_tiles, kbt, G, stages, wide;
  long long T;
  uint32_t tmem_cols;
  size_t smem, counters_bytes, partial_bytes;
};

Plan plan(int M, int N, int K, int nsm, bool has_lo) {
  Plan p{};
  // Token rows per tile: up to 256, but 128 with hi/lo activation pairs, so that
  // one MMA of N = 2 MT <= 256 covers both halves and a stage (weight box plus
  // two activation boxes, 48 KB) leaves room for four or more stages (a 256-row
  // pair tile took 80 KB stages, two of them, and measured 3-7x slower at 244 rows).
  const int mt_max = has_lo ? 128 : 256;
  p.MT = M > mt_max ? mt_max : ((M + 31) / 32) * 32;
  if (p.MT < 32) p.MT = 32;
  p.m_chunks = (M + p.MT - 1) / p.MT;
  p.n_tiles = N / kTileN;
  p.kbt = K / kBK;
  p.T = (long long)p.n_tiles * p.kbt;
  // Stream-K whenever the token rows fit in a few chunks (every weight-streaming
  // case, including the LM head); plain one-tile-per-CTA for large prefills.
  const bool split = p.m_chunks <= 4 || (long long)p.m_chunks * p.n_tiles < 2LL * nsm;
  p.G = split ? (int)std::min<long long>(nsm, p.T) : p.n_tiles;
  p.wide = has_lo && 2 * p.MT <= 256;
  uint32_t cols = 32;
  while (cols < (uint32_t)(2 * (p.wide ? 2 * p.MT : p.MT))) cols <<= 1;
  p.tmem_cols = cols;
  const size_t stage = kWBytes + (size_t)p.MT * kBK * 2 * (has_lo ? 2 : 1);
  const size_t fixed = (size_t)kSub * kLdt * 4 + kEpiRowSmemFloats * 4 + (2 * kMaxStages + 5) * 8 + 16 + 1024;
  int st = (int)((kSmemBudget - fixed) / stage);
  p.stages = std::max(2, std::min(kMaxStages, st));
  p.smem = (size_t)p.stages * stage + fixed;
  p.counters_bytes = kCounterBytes;
  p.partial_bytes = split ? (size_t)p.m_chunks * p.G * 2 * p.MT * kTileN * 4 : 0;
  return p;
}

}  // namespace

size_t gemm_tc_scratch_bytes(int M, int N, int K) {
  // enough for any M' <= M on up to kNsmSizing SMs, with or without hi/lo pairs
  size_t best = kCounterBytes;
  for (int lo = 0; lo < 2; ++lo) {
    const int mt = lo ? 128 : 256;
    const int chunks = (M + mt - 1) / mt;
    for (int mc = 1; mc <= chunks; ++mc) {
      const int Mp = mc == 1 ? std::min(M, mt) : mc * mt;
      const Plan p = plan(Mp, N, K, kNsmSizing, lo != 0);
      best = std::max(best, p.counters_bytes + p.partial_bytes);
    }
  }
  return best;
}

cudaError_t gemm_tc(const bf16* X, const bf16* X_lo, const bf16* W, int M, int N, int K, const EpiParams& ep,
                    void* scratch, int* status, cudaStream_t s, bool w_dep) {
  if (M <= 0) return cudaSuccess;
  if (N % kTileN || K % kBK || !scratch) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(X_lo) | reinterpret_cast<uintptr_t>(W)) & 15)
    return cudaErrorInvalidValue;
  const Plan p = plan(M, N, K, num_sms(), X_lo != nullptr);
  if ((long long)p.m_chunks * p.n_tiles > kCounterInts) return cudaErrorInvalidValue;
  CUtensorMap tmW, tmX, tmXlo;
  if (!make_tmap_bf16(&tmW, W, N, K, kTileN) || !make_tmap_bf16(&tmX, X, M, K, p.MT)) return cudaErrorInvalidValue;
  if (X_lo && !make_tmap_bf16(&tmXlo, X_lo, M, K, p.MT)) return cudaErrorInvalidValue;
  if (!X_lo) tmXlo = tmX;  // unused
  if (!raise_smem_limit(reinterpret_cast<const void*>(gemm_tc_kernel), kSmemBudget)) return cudaErrorInvalidValue;
  TcArgs a{};
  a.M = M;
  a.MT = p.MT;
  a.m_chunks = p.m_chunks;
  a.n_tiles = p.n_tiles;
  a.kbt = p.kbt;
  a.G = p.G;
  a.stages = p.stages;
  a.T = p.T;
  a.tmem_cols = p.tmem_cols;
  a.has_lo = X_lo != nullptr;
  a.wide = p.wide;
  a.w_dep = w_dep ? 1 : 0;
  a.counters = reinterpret_cast<int*>(scratch);
  a.partial = reinterpret_cast<float*>(reinterpret_cast<char*>(scratch) + p.counters_bytes);
  a.status = status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G * p.m_chunks);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel, tmW, tmX, tmXlo, a, ep);
}

}  // namespace eg

// ------------------------------------------------------------------ allocation-free entry point
//
// Some callers of the GEMM cannot allocate device memory: plugins of a host
// framework that owns the device allocator and does not let them call
// cudaMalloc, and code whose device-memory budget is fixed by someone else with
// no room for a scratch buffer. eagle_op_gemm_noalloc gives them the same tcgen05 kernel with
// its split-K scratch (arrival counters, then partial sums) in the static
// device array below instead of a caller buffer. The array is
// g_noalloc_scratch_bytes = 512 KiB of counters + 10 MiB of partials (160 SMs
// x 2 fragments x 64 rows x 128 columns x 4 bytes); every GPU that loads this
// library reserves it until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[eg::kNoAllocScratchBytes];

namespace eg {
namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_addr[256] = {};  // device address of g_noalloc_scratch, per device ordinal
}  // namespace
}  // namespace eg

extern "C" eagle_status eagle_op_gemm_noalloc(int32_t M, int32_t N, int32_t K, const void* d_x, const void* d_w,
                                              float* d_y, void* stream) {
  using namespace eg;
  if (M < 1 || N < 1 || K < 1 || !d_x || !d_w || !d_y) return EAGLE_ERR_INVALID_ARG;
  if (M > kNoAllocMaxM || N % kTileN || K % kBK || N / kTileN > kCounterInts) return EAGLE_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return EAGLE_ERR_CUDA;
  void* scratch = nullptr;
  {
    // first call on a device: look up the array's device address (host code
    // cannot use the symbol itself, which names a host-side shadow)
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return EAGLE_ERR_CUDA;
      g_noalloc_addr[dev] = p;
    }
    scratch = g_noalloc_addr[dev];
  }
  cudaStream_t s = (cudaStream_t)stream;
  // the array keeps the previous call's contents: the counters this shape uses must start at zero
  if (cudaMemsetAsync(scratch, 0, (size_t)(N / kTileN) * sizeof(int), s) != cudaSuccess) return EAGLE_ERR_CUDA;
  EpiParams e;
  e.kind = kEpiStore;
  e.M = M;
  e.N = N;
  e.y = d_y;
  const cudaError_t err = gemm_tc((const bf16*)d_x, nullptr, (const bf16*)d_w, M, N, K, e, scratch, nullptr, s);
  return err == cudaSuccess ? EAGLE_OK : (err == cudaErrorInvalidValue ? EAGLE_ERR_UNSUPPORTED : EAGLE_ERR_CUDA);
}

extern "C" eagle_status eagle_selftest_bounded_wait(int32_t* d_status, void* stream) {
  if (!d_status) return EAGLE_ERR_INVALID_ARG;
  eg::bounded_wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(d_status);
  return cudaGetLastError() == cudaSuccess ? EAGLE_OK : EAGLE_ERR_CUDA;
}
