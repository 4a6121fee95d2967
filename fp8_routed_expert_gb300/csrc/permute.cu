// Counting sort of the T*k (token, expert) pairs by expert.
//
// Trochilus ("Acknowledgements", the ds4 row) sorts (token, expert) pairs with
// a counting sort; the DeepSeek-V4.1-Flash post (§v3, "a short path for one
// token") shows why the per-expert token lists must be built on the device:
// finding them with a host round trip per expert stalls the copy stream.
//
// One CTA of 1024 threads: warp w owns the contiguous pair range
// [w*P/32, (w+1)*P/32).
//   1. per-warp histograms in shared memory,
//   2. per expert, an exclusive scan over the 32 warps gives each warp's base
//      inside the expert's segment; a block scan over experts gives offsets,
//   3. each warp scatters its range in ascending p, ranking equal experts
//      inside each 32-pair step with __match_any_sync,
// so every segment lists its pairs in ascending p (a stable sort) and the
// result is the same on every run.  Also emits the active-expert list, the
// per-expert count of 128-row tiles (for the grouped GEMM) and clears the
// per-position maxima the GEMV path accumulates.
#include "common.cuh"
#include "kernels.h"

namespace fp8moe {

__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_tot, int *total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int w = (lane < (int)(blockDim.x >> 5)) ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  int r = warp_tot[wid] + incl - v;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(1024) permute_kernel(
    const int32_t *__restrict__ idx, int64_t P, int E, int tile_m, int32_t *__restrict__ counts,
    int32_t *__restrict__ offsets, int32_t *__restrict__ perm, int32_t *__restrict__ inv,
    int32_t *__restrict__ active, int32_t *__restrict__ n_active,
    int32_t *__restrict__ tile_offsets, uint32_t *__restrict__ pos_max,
    int32_t *__restrict__ counters, int n_counters, int *__restrict__ err) {
  extern __shared__ int sm[];
  int *whist = sm;                 // [32][E]
  int *seg = sm + 32 * E;          // [E+1] segment starts
  __shared__ int warp_tot[32];
  __shared__ int total;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

  for (int i = tid; i < 32 * E; i += blockDim.x) whist[i] = 0;
  if (tid < n_counters) counters[tid] = 0;
  if (pos_max != nullptr)
    for (int64_t p = tid; p < P; p += blockDim.x) pos_max[p] = 0u;
  __syncthreads();

  const int64_t chunk = (P + 31) / 32;
  const int64_t p_lo = (int64_t)wid * chunk;
  const int64_t p_hi = (p_lo + chunk < P) ? p_lo + chunk : P;
  for (int64_t p = p_lo + lane; p < p_hi; p += 32) {
    int e = idx[p];
    if ((unsigned)e >= (unsigned)E) { set_error(err, DEV_ERR_BOUNDS); e = 0; }
    atomicAdd(&whist[wid * E + e], 1);
  }
  __syncthreads();

  // per expert: exclusive scan over warps (whist becomes the warp's base)
  for (int e = tid; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      int c = whist[w * E + e];
      whist[w * E + e] = run;
      run += c;
    }
    seg[e] = run;  // count, scanned below
  }
  __syncthreads();

  // block scans over experts (E <= 1024 = blockDim.x): offsets, active list, tiles
  {
    const int e = tid;
    const int c = (e < E) ? seg[e] : 0;
    const int off = block_exclusive_scan(c, warp_tot, &total);
    const int act = block_exclusive_scan(c > 0 ? 1 : 0, warp_tot, &total);
    const int nact = total;
    const int tiles = (c + tile_m - 1) / tile_m;
    const int toff = block_exclusive_scan(tiles, warp_tot, &total);
    const int ntiles = total;
    if (e < E) {
      counts[e] = c;
      offsets[e] = off;
      tile_offsets[e] = toff;
      if (c > 0) active[act] = e;
      seg[e] = off;
    }
    if (e == 0) {
      offsets[E] = (int32_t)P;
      tile_offsets[E] = ntiles;
      *n_active = nact;
    }
  }
  __syncthreads();

  // stable scatter
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int64_t base = p_lo; base < p_hi; base += 32) {
    const int64_t p = base + lane;
    const bool valid = p < p_hi;
    int e = valid ? idx[p] : -1;
    if (valid && (unsigned)e >= (unsigned)E) e = 0;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (valid) {
      const int rank = __popc(peers & lt_mask);
      const int pos = seg[e] + whist[wid * E + e] + rank;
      perm[pos] = (int32_t)p;
      inv[p] = pos;
    }
    __syncwarp();
    if (valid && (peers & lt_mask) == 0) whist[wid * E + e] += __popc(peers);
    __syncwarp();
  }
}

size_t permute_smem(int E) { return (size_t)(33 * E + 1) * sizeof(int); }

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
