// Counting sort of the T*k (token, expert) pairs by expert.
//
// Trochilus ("Acknowledgements", the ds4 row) sorts (token, expert) pairs with
// a counting sort; the DeepSeek-V4.1-Flash post (§v3, "a short path for one
// token") shows why the per-expert token lists must be built on the device:
// finding them with a host round trip per expert stalls the copy stream.
//
// One CTA: warp w owns the contiguous pair range [w*P/NW, (w+1)*P/NW).
//   1. per-warp histograms in shared memory,
//   2. per expert, an exclusive scan over the warps gives each warp's base
//      inside the expert's segment; block scans over experts give offsets,
//      the active-expert list and the per-expert 128-row tile offsets,
//   3. each warp scatters its range in ascending p, ranking equal experts
//      inside each 32-pair step with __match_any_sync,
// so every segment lists its pairs in ascending p (a stable sort) and the
// result is the same on every run.
#include "common.cuh"
#include "kernels.h"
#include "permute.cuh"

namespace fp8moe {

__global__ void __launch_bounds__(1024) permute_kernel(
    const int32_t *__restrict__ idx, int64_t P, int E, int tile_m, int32_t *__restrict__ counts,
    int32_t *__restrict__ offsets, int32_t *__restrict__ perm, int32_t *__restrict__ inv,
    int32_t *__restrict__ active, int32_t *__restrict__ n_active,
    int32_t *__restrict__ tile_offsets, uint32_t *__restrict__ pos_max,
    int32_t *__restrict__ counters, int n_counters, int *__restrict__ err) {
  extern __shared__ int sm[];
  for (int i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0;
  if (pos_max != nullptr)
    for (int64_t p = threadIdx.x; p < P; p += blockDim.x) pos_max[p] = 0u;
  SortOut o{counts, offsets, perm, inv, active, n_active, tile_offsets};
  cta_counting_sort<32>(idx, P, E, tile_m, o, sm, err);
}

size_t permute_smem(int E) { return cta_sort_smem(32, E); }

cudaError_t launch_permute(const int32_t *idx, int64_t P, int E, int tile_m, int32_t *counts,
                           int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *active,
                           int32_t *n_active, int32_t *tile_offsets, uint32_t *pos_max,
                           int32_t *counters, int n_counters, int *err, cudaStream_t s) {
  const size_t smem = permute_smem(E);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(permute_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  permute_kernel<<<1, 1024, smem, s>>>(idx, P, E, tile_m, counts, offsets, perm, inv, active,
                                       n_active, tile_offsets, pos_max, counters, n_counters, err);
  return cudaGetLastError();
}

}  // namespace fp8moe
