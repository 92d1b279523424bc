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
  // (fields read once: the shared-memory stores below may otherwise force reloads of p)
  const float* const ssq_in = p.ssq_in;
  const int n_ssq = p.n_ssq_in, M = p.M, kind = p.kind;
  const float inv_d = p.inv_d_in, eps = p.eps;
  const int* const rpos = p.rows.pos;
  const int* const rslot = p.rows.slot;
  const int* const rseq = p.rows.seq;
  const bool sampling = kind == kEpiLmHead && p.inv_temp > 0.f;
  const int* const spos = p.samp_pos;
  const int* const sseq = p.samp_seq;
  const int* const sidx = p.samp_idx;
  for (int m = tid; m < msub; m += nthr) {
    float sc = 1.f;
    if (ssq_in) {
      const float* s_in = ssq_in + m0 + m;
      float part[kEpiBatch];
#pragma unroll
      for (int q = 0; q < kEpiBatch; ++q) part[q] = 0.f;
      const int nfull = n_ssq - n_ssq % kEpiBatch;
      int j = 0;
      for (; j + 4 * kEpiBatch <= nfull; j += 4 * kEpiBatch) {
        float v[4 * kEpiBatch];
#pragma unroll
        for (int q = 0; q < 4 * kEpiBatch; ++q) v[q] = __ldcg(s_in + (size_t)(j + q) * M);
#pragma unroll
        for (int q = 0; q < 4 * kEpiBatch; ++q) part[q % kEpiBatch] += v[q];
      }
      for (; j < nfull; j += kEpiBatch) {
#pragma unroll
        for (int q = 0; q < kEpiBatch; ++q) part[q] += __ldcg(s_in + (size_t)(j + q) * M);
      }
      for (; j < n_ssq; ++j) part[0] += __ldcg(s_in + (size_t)j * M);
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < kEpiBatch; ++q) s += part[q];
      sc = rsqrtf(s * inv_d + eps);
    }
    r.scale[m] = sc;
    if (kind == kEpiQkv) {
      r.pos[m] = rpos[m0 + m];
      r.slot[m] = rslot[m0 + m];
      r.seq[m] = rseq[m0 + m];
    } else if (sampling) {  // the position of the token this row chooses, and its sequence
      const int src = sidx ? sidx[m0 + m] : m0 + m;
      r.pos[m] = spos[src] + 1;
      r.seq[m] = sseq[src];
    }
  }
}

// Four neighbouring elements of a staged tile row (one 16-byte access when the
// leading dimension keeps them aligned).
__device__ __forceinline__ float4 ld_tile4(const float* p, int ldt) {
  if ((ldt & 3) == 0) return *reinterpret_cast<const float4*>(p);
  return make_float4(p[0], p[1], p[2], p[3]);
}
__device__ __forceinline__ void st_tile4(float* p, int ldt, float4 v) {
  if ((ldt & 3) == 0) {
    *reinterpret_cast<float4*>(p) = v;
  } else {
    p[0] = v.x; p[1] = v.y; p[2] = v.z; p[3] = v.w;
  }
}
// The epilogue proper, with the row inputs already in r (visible to all 128
// threads); msub <= kEpiRows. Run by 128 threads with ranks tid = 0..127; sync()
// must be a barrier over exactly those threads.
template <typename T, typename Sync>
__device__ void epilogue_body(const EpiParams& p, float* tile, int ldt, int m0, int msub, int n0, EpiRows r,
                              int tid, Sync sync) {
  // Every field is read once into a register: the global stores below could
  // otherwise force the compiler to reload p's fields after each of them.
  const int kind = p.kind, M = p.M, N = p.N;
  const int ncols = min(kTileN, N - n0);
  float* const y = p.y;
  void* const out = p.out;
  bf16* const out_lo = p.out_lo;
  bf16* const hb_lo = p.hb_lo;
  const int q_dim = p.q_dim, kv_dim = p.kv_dim, head_dim = p.head_dim, n_kv = p.n_kv, cap = p.cap;
  const float* const rope_cos = p.rope_cos;
  const float* const rope_sin = p.rope_sin;
  void* const kc = p.kc;
  void* const vc = p.vc;
  __half* const qg = p.qg;
  const float qg_scale = p.qg_scale;
  const int ffn = p.ffn;
  float* const h = p.h;
  void* const hb = p.hb;
  float* const ssq_out = p.ssq_out;
  const float* const gain = p.gain;
  float* const h_tap = p.h_tap;
  float* const h_tap2 = p.h_tap2;
  const int topk = p.topk;
  const float inv_temp = p.inv_temp;
  const unsigned long long seed = p.seed;
  float* const rec_val = p.rec_val;
  int* const rec_idx = p.rec_idx;
  float* const rec_max = p.rec_max;
  float* const rec_sum = p.rec_sum;
  const float* rscale = r.scale;
  const int* rpos = r.pos;
  const int* rslot = r.slot;
  const int* rseq = r.seq;
  switch (kind) {
    case kEpiStore: {
      for (int m = 0; m < msub; ++m)
        if (tid < ncols) y[(size_t)(m0 + m) * N + n0 + tid] = tile[m * ldt + tid] * rscale[m];
      break;
    }
    case kEpiQkv: {
      // thread: columns c .. c + 3 (c = 4 (tid % 32)) of rows tid / 32, tid / 32 + 4, ...:
      // every access carries four neighbouring elements (a tile of 128 columns
      // holds whole head halves, so the four share their head, region and half).
      // The epilogue of a split tile's ~20-row slice is on the phase's critical
      // path: QKV phase 19.0 us per layer of the 8B verify with one column a
      // thread, 17.5 with two, 16.5 with four (fewer store instructions; the staged
      // tile's rows are 16-byte aligned for one shared-memory access per four).
      const int c = 4 * (tid & 31), rg = tid >> 5;
      if (c < ncols) {
        const int n = n0 + c;
        const int hd = head_dim, half = hd >> 1;
        const int i = n % hd;
        const int region = n < q_dim ? 0 : (n < q_dim + kv_dim ? 1 : 2);
        const int partner = i < half ? c + half : c - half;
        const int fi = i < half ? i : i - half;
        const int nn = n - q_dim - (region == 2 ? kv_dim : 0);
        const int kvh = nn / hd;
        __half* qgc = nullptr;
        int qg_row = 0;
        if (region == 0 && qg) {
          const int qh = n / hd, G = q_dim / hd / n_kv;
          qgc = qg + ((size_t)(qh / G) * M * G + qh % G) * hd + i;
          qg_row = G * hd;
        }
        constexpr int kB = kEpiLoadBatch / 4;  // rows of one batch for this thread
        for (int mb = rg; mb < msub; mb += 4 * kB) {
          float4 cs[kB], sn[kB];
#pragma unroll
          for (int q = 0; q < kB; ++q) {  // the batch's table loads, all in flight together
            cs[q] = make_float4(1.f, 1.f, 1.f, 1.f);
            sn[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (region < 2 && mb + 4 * q < msub) {
              const size_t at = (size_t)rpos[mb + 4 * q] * half + fi;
              cs[q] = *reinterpret_cast<const float4*>(rope_cos + at);
              sn[q] = *reinterpret_cast<const float4*>(rope_sin + at);
            }
          }
#pragma unroll
          for (int q = 0; q < kB; ++q) {
            const int m = mb + 4 * q;
            if (m >= msub) break;
            const float rs = rscale[m];
            float4 v = ld_tile4(tile + m * ldt + c, ldt);
            v.x *= rs; v.y *= rs; v.z *= rs; v.w *= rs;
            if (region < 2) {
              float4 pv = ld_tile4(tile + m * ldt + partner, ldt);
              const float sg = i < half ? -1.f : 1.f;
              v.x = v.x * cs[q].x + sg * (pv.x * rs) * sn[q].x;
              v.y = v.y * cs[q].y + sg * (pv.y * rs) * sn[q].y;
              v.z = v.z * cs[q].z + sg * (pv.z * rs) * sn[q].z;
              v.w = v.w * cs[q].w + sg * (pv.w * rs) * sn[q].w;
            }
            if (region == 0) {
              if (out) *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + (size_t)(m0 + m) * q_dim + n) = v;
              if (qgc) {
                __half2 a = __floats2half2_rn(v.x * qg_scale, v.y * qg_scale);
                __half2 b = __floats2half2_rn(v.z * qg_scale, v.w * qg_scale);
                uint2 u;
                u.x = *reinterpret_cast<uint32_t*>(&a);
                u.y = *reinterpret_cast<uint32_t*>(&b);
                *reinterpret_cast<uint2*>(qgc + (size_t)(m0 + m) * qg_row) = u;
              }
            } else if (rslot[m] >= 0) {
              const size_t at = (((size_t)rseq[m] * n_kv + kvh) * cap + rslot[m]) * hd + i;
              using KvT = typename KvOf<T>::type;
              KvT* const dst = reinterpret_cast<KvT*>(region == 1 ? kc : vc) + at;
              dst[0] = kv_from_f<T>(v.x);
              dst[1] = kv_from_f<T>(v.y);
              dst[2] = kv_from_f<T>(v.z);
              dst[3] = kv_from_f<T>(v.w);
            }
          }
        }
      }
      break;
    }
    case kEpiSwiglu: {
      const int blk = n0 / kTileN;
      const int rr = min(64, ffn - blk * 64);
      const int c = tid & 63;  // two threads per output column, on alternate rows
      if (c < rr) {
#pragma unroll 4
        for (int m = tid >> 6; m < msub; m += 2) {
          const float g = tile[m * ldt + c] * rscale[m];
          const float u = tile[m * ldt + rr + c] * rscale[m];
          store_hilo<T>(reinterpret_cast<T*>(out), out_lo, (size_t)(m0 + m) * ffn + blk * 64 + c, silu_f(g) * u);
        }
      }
      break;
    }
    case kEpiResid:
    case kEpiFc: {
      // thread: columns c .. c + 3 of rows tid / 32, tid / 32 + 4, ... (as in the QKV case)
      const int c = 4 * (tid & 31), rg = tid >> 5;
      if (c < ncols) {
        const int n = n0 + c;
        const float4 gn = *reinterpret_cast<const float4*>(gain + n);
        constexpr int kB = kEpiLoadBatch / 4;
        for (int mb = rg; mb < msub; mb += 4 * kB) {
          float4 hv[kB];
#pragma unroll
          for (int q = 0; q < kB; ++q)  // residual loads of the batch, ahead of its stores
            hv[q] = (kind == kEpiResid && mb + 4 * q < msub)
                        ? __ldcg(reinterpret_cast<const float4*>(h + (size_t)(m0 + mb + 4 * q) * N + n))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int q = 0; q < kB; ++q) {
            const int m = mb + 4 * q;
            if (m >= msub) break;
            const size_t at = (size_t)(m0 + m) * N + n;
            const float rs = rscale[m];
            const float4 t4 = ld_tile4(tile + m * ldt + c, ldt);
            const float4 hn = make_float4(hv[q].x + t4.x * rs, hv[q].y + t4.y * rs, hv[q].z + t4.z * rs,
                                          hv[q].w + t4.w * rs);
            *reinterpret_cast<float4*>(h + at) = hn;
            if (h_tap) *reinterpret_cast<float4*>(h_tap + at) = hn;
            if (h_tap2) *reinterpret_cast<float4*>(h_tap2 + at) = hn;
            store_hilo4<T>(reinterpret_cast<T*>(hb), hb_lo, at,
                           make_float4(hn.x * gn.x, hn.y * gn.y, hn.z * gn.z, hn.w * gn.w));
            st_tile4(tile + m * ldt + c, ldt, make_float4(hn.x * hn.x, hn.y * hn.y, hn.z * hn.z, hn.w * hn.w));
          }
        }
      } else {
        for (int m = rg; m < msub; m += 4) st_tile4(tile + m * ldt + c, ldt, make_float4(0.f, 0.f, 0.f, 0.f));
      }
      sync();
      const int warp = tid >> 5, lane = tid & 31;
      for (int m = warp; m < msub; m += 4) {
        float s = tile[m * ldt + lane] + tile[m * ldt + lane + 32] + tile[m * ldt + lane + 64] +
                  tile[m * ldt + lane + 96];
        s = warp_sum(s);
        if (lane == 0) ssq_out[(size_t)(n0 / kTileN) * M + m0 + m] = s;
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
          if (y && c < ncols) y[(size_t)(m0 + m) * N + n0 + c] = v[j];
          // sampling: the records (and so the merged top-1) are of the perturbed values
          if (inv_temp > 0.f && c < ncols) v[j] = v[j] * inv_temp + sample_gumbel(seed, rseq[m], rpos[m], n0 + c);
        }
        float mx = warp_max(fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])));
        float se = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) se += (lane + 32 * j < ncols) ? __expf(v[j] - mx) : 0.f;
        se = warp_sum(se);
        const size_t rec = (size_t)ti * M + m0 + m;
        if (lane == 0) {
          rec_max[rec] = mx;
          rec_sum[rec] = se;
        }
        for (int k = 0; k < topk; ++k) {
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
            rec_val[rec * topk + k] = wv;
            rec_idx[rec * topk + k] = wi < N ? wi : -1;
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
