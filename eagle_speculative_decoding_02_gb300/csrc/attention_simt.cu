// Tree-masked attention, SIMT form (float32 model path).
//
// A query row of group g sees the fully visible prefix slots [0, prefix) and
// slot prefix + i of the group's tree block for every bit i of its mask
// ("EAGLE (LLM decoding)", section "How EAGLE works": tree attention verifies
// all nodes in one forward pass). Keys are visited in slot order with an
// online (max-rescaled) softmax.
#include "kernels.h"

namespace eg {
namespace {

template <typename T>
__global__ void __launch_bounds__(128) attn_simt_kernel(AttnArgs a) {
  extern __shared__ float qs[];  // [4 warps][hd]
  const Group g = a.groups[blockIdx.x];
  const int h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hd = a.hd, nd = hd / 32;
  const int kvh = h * a.Hkv / a.Hq;
  const T* K = reinterpret_cast<const T*>(a.kc) + ((size_t)g.seq * a.Hkv + kvh) * a.cap * hd;
  const T* V = reinterpret_cast<const T*>(a.vc) + ((size_t)g.seq * a.Hkv + kvh) * a.cap * hd;
  float* q = qs + warp * hd;
  const int nkeys = g.prefix + g.block_len;
  for (int r = warp; r < g.nrows; r += 4) {
    const int row = g.row0 + r;
    const float* qr = a.q + ((size_t)row * a.Hq + h) * hd;
    for (int dd = lane; dd < hd; dd += 32) q[dd] = qr[dd];
    __syncwarp();
    const uint64_t m0 = a.mask[2 * row], m1 = a.mask[2 * row + 1];
    float mrun = -INFINITY, l = 0.f;
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k0 = 0; k0 < nkeys; k0 += 32) {
      const int j = k0 + lane;
      bool vis = false;
      if (j < g.prefix) {
        vis = true;
      } else if (j < nkeys) {
        const int b = j - g.prefix;
        vis = ((b < 64 ? (m0 >> b) : (m1 >> (b - 64))) & 1ull) != 0;
      }
      float s = -INFINITY;
      if (vis) {
        const T* kr = K + (size_t)j * hd;
        float acc = 0.f;
        for (int dd = 0; dd < hd; ++dd) acc = fmaf(q[dd], to_f(kr[dd]), acc);
        s = acc * a.scale;
      }
      const float cmax = warp_max(s);
      if (cmax == -INFINITY) continue;
      const float mnew = fmaxf(mrun, cmax);
      const float corr = __expf(mrun - mnew);
      const float pj = vis ? __expf(s - mnew) : 0.f;
      l = l * corr + warp_sum(pj);
      for (int i = 0; i < nd; ++i) o[i] *= corr;
      const int nk = min(32, nkeys - k0);
      for (int jj = 0; jj < nk; ++jj) {
        const float pb = __shfl_sync(0xffffffffu, pj, jj);
        if (pb != 0.f) {
          const T* vr = V + (size_t)(k0 + jj) * hd;
          for (int i = 0; i < nd; ++i) o[i] = fmaf(pb, to_f(vr[lane + 32 * i]), o[i]);
        }
      }
      mrun = mnew;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    T* orow = reinterpret_cast<T*>(a.o) + ((size_t)row * a.Hq + h) * hd;
    for (int i = 0; i < nd; ++i) orow[lane + 32 * i] = from_f<T>(o[i] * inv);
    __syncwarp();
  }
}

}  // namespace

template <typename T>
cudaError_t attention_simt(const AttnArgs& a, cudaStream_t s) {
  if (a.n_groups <= 0) return cudaSuccess;
  if (a.hd % 32 != 0 || a.hd > 128) return cudaErrorInvalidValue;
  dim3 grid(a.n_groups, a.Hq);
  attn_simt_kernel<T><<<grid, 128, 4 * a.hd * sizeof(float), s>>>(a);
  return cudaGetLastError();
}

template cudaError_t attention_simt<float>(const AttnArgs&, cudaStream_t);

}  // namespace eg
