// Stable counting sort of (token, expert) pairs by expert: CTA-wide (the
// standalone permutation kernel) and one-warp (the small-batch routing).
#pragma once

#include "common.cuh"

namespace fp8moe {

struct SortOut {
  int32_t *counts, *offsets, *perm, *inv, *active, *n_active, *tile_offsets;
};

// Shared memory (bytes) of cta_counting_sort with NW warps and E experts.
__host__ __device__ inline size_t cta_sort_smem(int NW, int E) { return (size_t)((NW + 1) * E + 1 + 64) * sizeof(int); }

// Exclusive scan of one int per thread over the CTA; *total gets the sum.
// Every thread of the CTA must call it.  tmp: >= 33 ints of shared memory.
__device__ __forceinline__ int cta_exclusive_scan(int v, int *tmp, int *total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) tmp[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int w = lane < nw ? tmp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    tmp[lane] = wi - w;
    if (lane == 31) tmp[32] = wi;
  }
  __syncthreads();
  const int r = tmp[wid] + incl - v;
  *total = tmp[32];
  __syncthreads();
  return r;
}

// Stable counting sort by expert of pairs p in [0, P) with experts idx[p],
// done by one CTA of NW warps.  smem: cta_sort_smem(NW, E) bytes.
template <int NW>
__device__ void cta_counting_sort(const int32_t *idx, int64_t P, int E, int tile_m,
                                  const SortOut &o, int *smem, int *err) {
  int *whist = smem;                 // [NW][E]
  int *seg = smem + NW * E;          // [E] segment starts
  int *tmp = seg + E + 1;            // scan scratch (>= 33)
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nt = blockDim.x;

  for (int i = tid; i < NW * E; i += nt) whist[i] = 0;
  __syncthreads();

  const int64_t chunk = (P + NW - 1) / NW;
  const int64_t p_lo = (int64_t)wid * chunk;
  const int64_t p_hi = (p_lo + chunk < P) ? p_lo + chunk : P;
  for (int64_t p = p_lo + lane; p < p_hi; p += 32) {
    int e = idx[p];
    if ((unsigned)e >= (unsigned)E) { set_error(err, DEV_ERR_BOUNDS); e = 0; }
    atomicAdd(&whist[wid * E + e], 1);
  }
  __syncthreads();

  // per expert: exclusive scan over warps (whist becomes each warp's base)
  for (int e = tid; e < E; e += nt) {
    int run = 0;
#pragma unroll 8
    for (int w = 0; w < NW; ++w) {
      const int c = whist[w * E + e];
      whist[w * E + e] = run;
      run += c;
    }
    seg[e] = run;  // count for now
  }
  __syncthreads();

  // scans over experts; thread t owns experts [t*per, (t+1)*per)
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
    seg[e] = off;
    off += c;
    toff += (c + tile_m - 1) / tile_m;
  }
  if (tid == 0) {
    o.offsets[E] = (int32_t)P;
    o.tile_offsets[E] = tot_t;
    *o.n_active = tot_a;
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
      o.perm[pos] = (int32_t)p;
      o.inv[p] = pos;
    }
    __syncwarp();
    if (valid && (peers & lt_mask) == 0) whist[wid * E + e] += __popc(peers);
    __syncwarp();
  }
}

// The same sort by ONE warp, for small P (the decode path's few hundred
// pairs): a compact code path matters more there than parallelism.  Every
// lane of the calling warp must call it; cur: E ints of shared memory.
__device__ __forceinline__ void warp_counting_sort(const int32_t *idx, int P, int E, int tile_m,
                                                   const SortOut &o, int *cur, int *err) {
  const int lane = threadIdx.x & 31;
  for (int e = lane; e < E; e += 32) cur[e] = 0;
  __syncwarp();
  for (int p = lane; p < P; p += 32) {
    int e = idx[p];
    if ((unsigned)e >= (unsigned)E) {
      set_error(err, DEV_ERR_BOUNDS);
      e = 0;
    }
    atomicAdd(&cur[e], 1);
  }
  __syncwarp();
  // lane l owns experts [l per, (l + 1) per): counts, then scans over lanes
  const int per = (E + 31) / 32, e0 = lane * per, e1 = e0 + per < E ? e0 + per : E;
  int c_sum = 0, a_sum = 0, t_sum = 0;
  for (int e = e0; e < e1; ++e) {
    const int c = cur[e];
    c_sum += c;
    a_sum += c > 0;
    t_sum += (c + tile_m - 1) / tile_m;
  }
  int c_inc = c_sum, a_inc = a_sum, t_inc = t_sum;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int c2 = __shfl_up_sync(0xffffffffu, c_inc, d), a2 = __shfl_up_sync(0xffffffffu, a_inc, d);
    const int t2 = __shfl_up_sync(0xffffffffu, t_inc, d);
    if (lane >= d) {
      c_inc += c2;
      a_inc += a2;
      t_inc += t2;
    }
  }
  int off = c_inc - c_sum, act = a_inc - a_sum, toff = t_inc - t_sum;
  for (int e = e0; e < e1; ++e) {
    const int c = cur[e];
    o.counts[e] = c;
    o.offsets[e] = off;
    o.tile_offsets[e] = toff;
    if (c > 0) o.active[act++] = e;
    cur[e] = off;  // becomes the expert's write cursor
    off += c;
    toff += (c + tile_m - 1) / tile_m;
  }
  if (lane == 31) {
    o.offsets[E] = P;
    o.tile_offsets[E] = t_inc;
    *o.n_active = a_inc;
  }
  __syncwarp();
  // stable scatter, 32 pairs at a time in pair order
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = 0; base < P; base += 32) {
    const int p = base + lane;
    const bool valid = p < P;
    int e = valid ? idx[p] : -1;
    if (valid && (unsigned)e >= (unsigned)E) e = 0;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (valid) {
      const int pos = cur[e] + rank;
      o.perm[pos] = p;
      o.inv[p] = pos;
    }
    __syncwarp();
    if (valid && rank == 0) cur[e] += __popc(peers);
    __syncwarp();
  }
}

}  // namespace fp8moe
