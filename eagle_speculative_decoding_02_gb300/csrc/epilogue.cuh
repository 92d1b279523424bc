// GEMM epilogues shared by the SIMT and the tcgen05 GEMM.
//
// Both GEMMs finish an output tile of up to 128 weight rows (columns n of Y)
// by `msub` token rows (rows m of Y) as float32 in shared memory,
// tile[m * ldt + c] = sum_k X[m0+m][k] W[n0+c][k], and call run_epilogue with
// 128 threads. The epilogue applies the RMSNorm row scale of the GEMM input
// and the op that follows the projection in a Llama decoder layer.
#pragma once

#include "common.cuh"

namespace eg {

// Rows per epilogue call, and the shared-memory row staging it needs:
// row scale, RoPE position, KV slot and sequence of each row.
constexpr int kEpiRows = 32;
constexpr int kEpiRowSmemFloats = 4 * kEpiRows;
// The row sum of squares is accumulated in kEpiBatch interleaved partial sums
// (fixed order); per-column loads of one thread (RoPE tables, residual) are
// issued kEpiLoadBatch rows at a time, ahead of any store, so that their
// latencies overlap.
constexpr int kEpiBatch = 8;
constexpr int kEpiLoadBatch = 16;

// Per-row inputs of an epilogue: the RMSNorm scale of the GEMM input row and,
// for the QKV epilogue, its RoPE position, KV slot and sequence. Entry m
// describes row m0 + m of the call.
struct EpiRows {
  float* scale;
  int* pos;
  int* slot;
  int* seq;
  __device__ EpiRows at(int off) const { return {scale + off, pos + off, slot + off, seq + off}; }
};
// Row arrays of `cap` rows carved out of 4 * cap words of shared memory.
__device__ inline EpiRows epi_rows(float* sm, int cap) {
  return {sm, reinterpret_cast<int*>(sm + cap), reinterpret_cast<int*>(sm + 2 * cap),
          reinterpret_cast<int*>(sm + 3 * cap)};
}

// Inputs that earlier phases of the same persistent launch may have written
// (row sums of squares, the residual stream) are read through L2 (ld.global.cg):
// the SM's L1 is not coherent with other SMs' stores within one launch.

// Fills r for rows m0 .. m0 + msub - 1; thread tid of nthr takes rows tid,
// tid + nthr, ... The row scale sums the input's column-tile partials j in
// partial sum j % kEpiBatch (complete batches), the rest into partial 0, then
// adds the partials in order; its loads are issued 32 at a time.
__device__ inline void load_epi_rows(const EpiParams& p, int m0, int msub, EpiRows r, int tid, int nthr) {
  for (int m = tid; m < msub; m += nthr) {
    float sc = 1.f;
    if (p.ssq_in) {
      const float* s_in = p.ssq_in + m0 + m;
      float part[kEpiBatch];
#pragma unroll
      for (int q = 0; q < kEpiBatch; ++q) part[q] = 0.f;
      const int nfull = p.n_ssq_in - p.n_ssq_in % kEpiBatch;
      int j = 0;
      for (; j + 4 * kEpiBatch <= nfull; j += 4 * kEpiBatch) {
        float v[4 * kEpiBatch];
#pragma unroll
        for (int q = 0; q < 4 * kEpiBatch; ++q) v[q] = __ldcg(s_in + (size_t)(j + q) * p.M);
#pragma unroll
        for (int q = 0; q < 4 * kEpiBatch; ++q) part[q % kEpiBatch] += v[q];
      }
      for (; j < nfull; j += kEpiBatch) {
#pragma unroll
        for (int q = 0; q < kEpiBatch; ++q) part[q] += __ldcg(s_in + (size_t)(j + q) * p.M);
      }
      for (; j < p.n_ssq_in; ++j) part[0] += __ldcg(s_in + (size_t)j * p.M);
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < kEpiBatch; ++q) s += part[q];
      sc = rsqrtf(s * p.inv_d_in + p.eps);
    }
    r.scale[m] = sc;
    if (p.kind == kEpiQkv) {
      r.pos[m] = p.rows.pos[m0 + m];
      r.slot[m] = p.rows.slot[m0 + m];
      r.seq[m] = p.rows.seq[m0 + m];
    }
  }
}

// The epilogue proper, with the row inputs already in r (visible to all 128
// threads); msub <= kEpiRows. Run by 128 threads with ranks tid = 0..127; sync()
// must be a barrier over exactly those threads.
template <typename T, typename Sync>
__device__ void epilogue_body(const EpiParams& p, float* tile, int ldt, int m0, int msub, int n0, EpiRows r,
                              int tid, Sync sync) {
  const int ncols = min(kTileN, p.N - n0);
  const float* rscale = r.scale;
  const int* rpos = r.pos;
  const int* rslot = r.slot;
  const int* rseq = r.seq;
  switch (p.kind) {
    case kEpiStore: {
      for (int m = 0; m < msub; ++m)
        if (tid < ncols) p.y[(size_t)(m0 + m) * p.N + n0 + tid] = tile[m * ldt + tid] * rscale[m];
      break;
    }
    case kEpiQkv: {
      const int c = tid;
      if (c < ncols) {
        const int n = n0 + c;
        const int hd = p.head_dim, half = hd >> 1;
        const int i = n % hd;
        const int region = n < p.q_dim ? 0 : (n < p.q_dim + p.kv_dim ? 1 : 2);
        const int partner = i < half ? c + half : c - half;
        const int fi = i < half ? i : i - half;
        const int nn = n - p.q_dim - (region == 2 ? p.kv_dim : 0);
        const int kvh = nn / hd;
        // this column's element of the grouped half queries, row 0
        __half* qgc = nullptr;
        int qg_row = 0;
        if (region == 0 && p.qg) {
          const int qh = n / hd, G = p.q_dim / hd / p.n_kv;
          qgc = p.qg + ((size_t)(qh / G) * p.M * G + qh % G) * hd + i;
          qg_row = G * hd;
        }
        for (int mb = 0; mb < msub; mb += kEpiLoadBatch) {
          float cs[kEpiLoadBatch], sn[kEpiLoadBatch];
#pragma unroll
          for (int q = 0; q < kEpiLoadBatch; ++q) {  // the batch's table loads, all in flight together
            cs[q] = 1.f;
            sn[q] = 0.f;
            if (region < 2 && mb + q < msub) {
              const size_t at = (size_t)rpos[mb + q] * half + fi;
              cs[q] = p.rope_cos[at];
              sn[q] = p.rope_sin[at];
            }
          }
#pragma unroll
          for (int q = 0; q < kEpiLoadBatch; ++q) {
            const int m = mb + q;
            if (m >= msub) break;
            float v = tile[m * ldt + c] * rscale[m];
            if (region < 2) {
              const float pv = tile[m * ldt + partner] * rscale[m];
              v = i < half ? v * cs[q] - pv * sn[q] : v * cs[q] + pv * sn[q];
            }
            if (region == 0) {
              reinterpret_cast<float*>(p.out)[(size_t)(m0 + m) * p.q_dim + n] = v;
              if (qgc) qgc[(size_t)(m0 + m) * qg_row] = __float2half_rn(v * p.qg_scale);
            } else if (rslot[m] >= 0) {
              const size_t at = (((size_t)rseq[m] * p.n_kv + kvh) * p.cap + rslot[m]) * hd + i;
              using KvT = typename KvOf<T>::type;
              reinterpret_cast<KvT*>(region == 1 ? p.kc : p.vc)[at] = kv_from_f<T>(v);
            }
          }
        }
      }
      break;
    }
    case kEpiSwiglu: {
      const int blk = n0 / kTileN;
      const int rr = min(64, p.ffn - blk * 64);
      const int c = tid & 63;  // two threads per output column, on alternate rows
      if (c < rr) {
#pragma unroll 4
        for (int m = tid >> 6; m < msub; m += 2) {
          const float g = tile[m * ldt + c] * rscale[m];
          const float u = tile[m * ldt + rr + c] * rscale[m];
          store_hilo<T>(reinterpret_cast<T*>(p.out), p.out_lo, (size_t)(m0 + m) * p.ffn + blk * 64 + c, silu_f(g) * u);
        }
      }
      break;
    }
    case kEpiResid:
    case kEpiFc: {
      const int c = tid;
      if (c < ncols) {
        const int n = n0 + c;
        const float gn = p.gain[n];
        for (int mb = 0; mb < msub; mb += kEpiLoadBatch) {
          float hv[kEpiLoadBatch];
#pragma unroll
          for (int q = 0; q < kEpiLoadBatch; ++q)  // residual loads of the batch, ahead of its stores
            hv[q] = (p.kind == kEpiResid && mb + q < msub) ? __ldcg(p.h + (size_t)(m0 + mb + q) * p.N + n) : 0.f;
#pragma unroll
          for (int q = 0; q < kEpiLoadBatch; ++q) {
            const int m = mb + q;
            if (m >= msub) break;
            const size_t at = (size_t)(m0 + m) * p.N + n;
            const float hn = hv[q] + tile[m * ldt + c] * rscale[m];
            p.h[at] = hn;
            store_hilo<T>(reinterpret_cast<T*>(p.hb), p.hb_lo, at, hn * gn);
            tile[m * ldt + c] = hn * hn;
          }
        }
      } else {
        for (int m = 0; m < msub; ++m) tile[m * ldt + c] = 0.f;
      }
      sync();
      const int warp = tid >> 5, lane = tid & 31;
      for (int m = warp; m < msub; m += 4) {
        float s = tile[m * ldt + lane] + tile[m * ldt + lane + 32] + tile[m * ldt + lane + 64] +
                  tile[m * ldt + lane + 96];
        s = warp_sum(s);
        if (lane == 0) p.ssq_out[(size_t)(n0 / kTileN) * p.M + m0 + m] = s;
      }
      break;
    }
    case kEpiLmHead: {
      const int warp = tid >> 5, lane = tid & 31;
      const int ti = n0 / kTileN;
      for (int m = warp; m < msub; m += 4) {
        float v[4];
        int idx[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = lane + 32 * j;
          idx[j] = n0 + c;
          v[j] = c < ncols ? tile[m * ldt + c] * rscale[m] : -INFINITY;
          if (p.y && c < ncols) p.y[(size_t)(m0 + m) * p.N + n0 + c] = v[j];
        }
        float mx = warp_max(fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])));
        float se = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) se += (lane + 32 * j < ncols) ? __expf(v[j] - mx) : 0.f;
        se = warp_sum(se);
        const size_t rec = (size_t)ti * p.M + m0 + m;
        if (lane == 0) {
          p.rec_max[rec] = mx;
          p.rec_sum[rec] = se;
        }
        for (int k = 0; k < p.topk; ++k) {
          float bv = v[0];
          int bi = idx[0], bj = 0;
#pragma unroll
          for (int j = 1; j < 4; ++j)
            if (v[j] > bv || (v[j] == bv && idx[j] < bi)) { bv = v[j]; bi = idx[j]; bj = j; }
          float wv = bv;
          int wi = bi;
          warp_argmax(wv, wi);
          if (bi == wi && bv == wv) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (j == bj) v[j] = -INFINITY;
          }
          if (lane == 0) {
            p.rec_val[rec * p.topk + k] = wv;
            p.rec_idx[rec * p.topk + k] = wi < p.N ? wi : -1;
          }
        }
      }
      break;
    }
  }
  sync();
}

// Loads the row inputs into rowsm (kEpiRowSmemFloats words), then runs the epilogue.
template <typename T, typename Sync>
__device__ void run_epilogue(const EpiParams& p, float* tile, int ldt, int m0, int msub, int n0,
                             float* rowsm, int tid, Sync sync) {
  const EpiRows r = epi_rows(rowsm, kEpiRows);
  load_epi_rows(p, m0, msub, r, tid, 128);
  sync();
  epilogue_body<T>(p, tile, ldt, m0, msub, n0, r, tid, sync);
}

}  // namespace eg
