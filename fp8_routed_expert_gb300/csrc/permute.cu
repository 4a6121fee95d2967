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

// ---------------------------------------------------------------- many CTAs
// For large P the same stable sort runs over kPermChunk-pair chunks, one CTA
// each (warp w of CTA c owns pairs [c kPermChunk + w kPermChunk / 8, + kPermChunk / 8)):
//   1. perm_hist_kernel: each chunk's count per expert -> chunk_hist[c][e];
//   2. perm_scan_kernel (one CTA): per expert an exclusive scan over the
//      chunks (chunk_hist becomes each chunk's base inside the segment), then
//      the scans over experts of the one-CTA sort;
//   3. perm_scatter_kernel: each chunk recounts per warp, scans over its warps
//      and scatters in ascending p as in the one-CTA sort.
// Segments list their pairs in ascending p, as with one CTA; the scattered
// stores and the histogram atomics spread over many SMs.
namespace {

constexpr int kPermWarps = 8;
constexpr int kPermChunk = 2048;

__device__ __forceinline__ void warp_range(int64_t P, int64_t &lo, int64_t &hi) {
  const int64_t c0 = (int64_t)blockIdx.x * kPermChunk, w = threadIdx.x >> 5;
  lo = c0 + w * (kPermChunk / kPermWarps);
  hi = lo + kPermChunk / kPermWarps;
  if (hi > P) hi = P;
}

// Per-warp counts of this CTA's chunk into whist [kPermWarps][E].
__device__ __forceinline__ void chunk_warp_hist(const int32_t *__restrict__ idx, int64_t P, int E,
                                                int *whist, int *err) {
  for (int i = threadIdx.x; i < kPermWarps * E; i += blockDim.x) whist[i] = 0;
  __syncthreads();
  int64_t lo, hi;
  warp_range(P, lo, hi);
  const int wid = threadIdx.x >> 5;
  for (int64_t p = lo + (threadIdx.x & 31); p < hi; p += 32) {
    int e = idx[p];
    if ((unsigned)e >= (unsigned)E) {
      set_error(err, DEV_ERR_BOUNDS);
      e = 0;
    }
    atomicAdd(&whist[wid * E + e], 1);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(32 * kPermWarps) perm_hist_kernel(const int32_t *__restrict__ idx, int64_t P,
                                                                   int E, int32_t *__restrict__ chunk_hist,
                                                                   uint32_t *__restrict__ pos_max,
                                                                   int32_t *__restrict__ counters,
                                                                   int n_counters, int *__restrict__ err) {
  extern __shared__ int whist[];
  pdl_wait();  // the experts come from the previous kernel
  pdl_trigger();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0;
  if (pos_max != nullptr) {
    const int64_t c0 = (int64_t)blockIdx.x * kPermChunk;
    for (int64_t p = c0 + threadIdx.x; p < c0 + kPermChunk && p < P; p += blockDim.x) pos_max[p] = 0u;
  }
  chunk_warp_hist(idx, P, E, whist, err);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int sum = 0;
#pragma unroll
    for (int w = 0; w < kPermWarps; ++w) sum += whist[w * E + e];
    chunk_hist[(int64_t)blockIdx.x * E + e] = sum;
  }
}

__global__ void __launch_bounds__(1024) perm_scan_kernel(int64_t P, int E, int n_chunks, int tile_m,
                                                         int32_t *__restrict__ chunk_hist, SortOut o) {
  extern __shared__ int sm[];
  int *seg = sm;          // [E] counts
  int *tmp = sm + E + 1;  // scan scratch (>= 33)
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int e = tid; e < E; e += nt) {
    int run = 0;
    for (int c = 0; c < n_chunks; ++c) {
      const int v = chunk_hist[(int64_t)c * E + e];
      chunk_hist[(int64_t)c * E + e] = run;
      run += v;
    }
    seg[e] = run;
  }
  __syncthreads();
  // scans over experts; thread t owns experts [t per, (t + 1) per)
  const int per = (E + nt - 1) / nt;
  const int e0 = tid * per;
  int c_sum = 0, a_sum = 0, t_sum = 0;
  for (int e = e0; e < e0 + per && e < E; ++e) {
    const int c = seg[e];
    c_sum += c;
    a_sum += c > 0;
    t_sum += (c + tile_m - 1) / tile_m;
  }
  int tot_c, tot_a, tot_t;
  int off = cta_exclusive_scan(c_sum, tmp, &tot_c);
  int act = cta_exclusive_scan(a_sum, tmp, &tot_a);
  int toff = cta_exclusive_scan(t_sum, tmp, &tot_t);
  for (int e = e0; e < e0 + per && e < E; ++e) {
    const int c = seg[e];
    o.counts[e] = c;
    o.offsets[e] = off;
    o.tile_offsets[e] = toff;
    if (c > 0) o.active[act++] = e;
    off += c;
    toff += (c + tile_m - 1) / tile_m;
  }
  if (tid == 0) {
    o.offsets[E] = (int32_t)P;
    o.tile_offsets[E] = tot_t;
    *o.n_active = tot_a;
  }
}

__global__ void __launch_bounds__(32 * kPermWarps) perm_scatter_kernel(const int32_t *__restrict__ idx,
                                                                      int64_t P, int E,
                                                                      const int32_t *__restrict__ chunk_base,
                                                                      SortOut o, int *__restrict__ err) {
  extern __shared__ int whist[];  // [kPermWarps][E]
  pdl_wait();
  pdl_trigger();
  chunk_warp_hist(idx, P, E, whist, err);
  // per expert: each warp's first position = segment start + the chunk's base
  // inside the segment + the earlier warps' counts
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = o.offsets[e] + chunk_base[(int64_t)blockIdx.x * E + e];
#pragma unroll
    for (int w = 0; w < kPermWarps; ++w) {
      const int c = whist[w * E + e];
      whist[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  int64_t lo, hi;
  warp_range(P, lo, hi);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int64_t base = lo; base < hi; base += 32) {
    const int64_t p = base + lane;
    const bool valid = p < hi;
    int e = valid ? idx[p] : -1;
    if (valid && (unsigned)e >= (unsigned)E) e = 0;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (valid) {
      const int pos = whist[wid * E + e] + __popc(peers & lt_mask);
      o.perm[pos] = (int32_t)p;
      o.inv[p] = pos;
    }
    __syncwarp();
    if (valid && (peers & lt_mask) == 0) whist[wid * E + e] += __popc(peers);
    __syncwarp();
  }
}

}  // namespace

int64_t permute_chunks(int64_t P) { return (P + kPermChunk - 1) / kPermChunk; }

cudaError_t launch_permute(const int32_t *idx, int64_t P, int E, int tile_m, int32_t *counts,
                           int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *active,
                           int32_t *n_active, int32_t *tile_offsets, uint32_t *pos_max,
                           int32_t *counters, int n_counters, int *err, cudaStream_t s,
                           int32_t *chunk_hist) {
  const int64_t n_chunks = permute_chunks(P);
  if (chunk_hist != nullptr && n_chunks > 2) {
    const SortOut o{counts, offsets, perm, inv, active, n_active, tile_offsets};
    const size_t hsmem = (size_t)kPermWarps * E * sizeof(int);
    cudaError_t e;
    if (hsmem > 48 * 1024) {
      if ((e = cudaFuncSetAttribute(perm_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hsmem)) !=
              cudaSuccess ||
          (e = cudaFuncSetAttribute(perm_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)hsmem)) != cudaSuccess)
        return e;
    }
    if ((e = launch_pdl(perm_hist_kernel, dim3((unsigned)n_chunks), dim3(32 * kPermWarps), hsmem, s, idx, P, E,
                        chunk_hist, pos_max, counters, n_counters, err)) != cudaSuccess)
      return e;
    if ((e = launch_pdl(perm_scan_kernel, dim3(1), dim3(1024), (size_t)(E + 1 + 64) * sizeof(int), s, P, E,
                        (int)n_chunks, tile_m, chunk_hist, o)) != cudaSuccess)
      return e;
    return launch_pdl(perm_scatter_kernel, dim3((unsigned)n_chunks), dim3(32 * kPermWarps), hsmem, s, idx, P,
                      E, static_cast<const int32_t *>(chunk_hist), o, err);
  }
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
