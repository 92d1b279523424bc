// Standalone tree-attention kernels (one work item per CTA, then a merge
// kernel); the bodies live in attention_tc.cuh.
#include "attention_tc.cuh"

namespace eg {
namespace {

using namespace attn;
// Keys per work item and per staging sub-chunk: the same as the persistent
// layer-stack kernel's, so that both paths sum every attention output in the
// same order (bit-identical rows).
constexpr int kCKI = 256;
constexpr int kCKS = 64;

template <int HD>
__global__ void __launch_bounds__(kAttnThreads) attn_tc_kernel(AttnArgs a, int n_chunk_slots) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  half* buf = reinterpret_cast<half*>(smem_raw);  // two staging buffers, each K then V
  // programmatic dependent launch: every CTA waits for the producer of q / K / V before any read
  pdl_wait();
  if (threadIdx.x == 0) pdl_trigger();
  attn_item<HD, kCKI, kCKS>(a, blockIdx.x, blockIdx.y, blockIdx.z, n_chunk_slots, buf, 2, threadIdx.x,
                            BlockSync{});
}

template <int HD>
__global__ void attn_merge_kernel(AttnArgs a, int n_chunk_slots) {
  pdl_wait();
  if (threadIdx.x == 0) pdl_trigger();
  const int w = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (w < a.M * a.Hq) attn_merge_warp<HD, kCKI>(a, w, threadIdx.x & 31, n_chunk_slots);
}

template <int HD>
cudaError_t launch(const AttnArgs& a, cudaStream_t s) {
  const int slots = n_prefix_chunks(a.max_prefix, kCKI) + 1;
  const size_t smem = 2 * smem_bytes<HD, kCKS>();  // double-buffered sub-chunks
  if (!raise_smem_limit(reinterpret_cast<const void*>(attn_tc_kernel<HD>), (int)smem)) return cudaErrorInvalidValue;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  const int rb_count = row_blocks(a.Hq, a.Hkv);
  cfg.gridDim = dim3(slots, a.Hkv * rb_count, a.n_groups);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_tc_kernel<HD>, a, slots);
  if (e != cudaSuccess) return e;
  const int warps = a.M * a.Hq;
  cfg.gridDim = dim3((warps + 3) / 4);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, attn_merge_kernel<HD>, a, slots);
}

}  // namespace

size_t attention_tc_scratch_bytes(int M, int Hq, int hd, int max_prefix) {
  const size_t slots = (size_t)n_prefix_chunks(max_prefix, kCKI) + 1;
  return (size_t)M * Hq * slots * (hd + 2) * sizeof(float);
}

cudaError_t attention_tc(const AttnArgs& a, cudaStream_t s) {
  if (a.n_groups <= 0 || a.M <= 0) return cudaSuccess;
  if (!a.part || a.Hq % a.Hkv) return cudaErrorInvalidValue;
  if (a.hd == 128) return launch<128>(a, s);
  if (a.hd == 64) return launch<64>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace eg
