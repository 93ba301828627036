// Pool staging copy (pic_stage_pool): the pool rows a batch reads, copied
// from a pool in pinned host memory into a device pool of the same layout by
// SM loads and stores over the host link (on GB300, NVLink-C2C to Grace
// memory).  Plain copy engines would do the same bytes, but a copy engine
// serves its queue in order: a stitch's small workspace upload queued behind
// gigabytes of pool copies waits for all of them, which defeats staging one
// request group while the previous one is stitched.
//   * Work item = one span (a range of pool rows of one layer, contiguous in
//     both pools) of one layer of one tensor (K or V); a grid of one CTA per
//     SM strides over the items.
//   * Each thread keeps 8 16-byte loads in flight (32 KB per CTA, about 5 MB
//     over the grid: far more than the link's bandwidth-latency product), with
//     streaming hints: the host rows are read once, the device rows are read
//     by the stitch that follows, not by this launch.
#include <cuda_runtime.h>

#include <cstdint>

#include "pic_internal.h"

namespace pic {
namespace {

constexpr int kStageThreads = 256;
constexpr int kStageUnroll = 8;

__global__ void __launch_bounds__(kStageThreads) k_stage_rows(const __grid_constant__ StageParams p) {
  const int64_t items = static_cast<int64_t>(p.tensors) * p.layers * p.n_spans;
  for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
    const int s = static_cast<int>(it % p.n_spans);
    const int64_t tl = it / p.n_spans;
    const int l = static_cast<int>(tl % p.layers), t = static_cast<int>(tl / p.layers);
    const StageSpan sp = p.spans[s];
    const uint4* src = reinterpret_cast<const uint4*>(p.src[t] + l * p.src_ls + sp.off);
    uint4* dst = reinterpret_cast<uint4*>(p.dst[t] + l * p.dst_ls + sp.off);
    const int64_t nv = sp.bytes >> 4;
    for (int64_t i = threadIdx.x; i < nv; i += static_cast<int64_t>(kStageUnroll) * kStageThreads) {
      uint4 v[kStageUnroll];
#pragma unroll
      for (int k = 0; k < kStageUnroll; ++k) {
        const int64_t j = i + static_cast<int64_t>(k) * kStageThreads;
        if (j < nv) v[k] = __ldcs(src + j);
      }
#pragma unroll
      for (int k = 0; k < kStageUnroll; ++k) {
        const int64_t j = i + static_cast<int64_t>(k) * kStageThreads;
        if (j < nv) __stcs(dst + j, v[k]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_stage_rows(const StageParams& p, int grid, cudaStream_t stream) {
  k_stage_rows<<<grid, kStageThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pic
