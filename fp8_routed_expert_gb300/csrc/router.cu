// Router: f32 logits, certified top-k selection and renormalised weights.
//
// The router reads f32 weights (dragon.c, "Precision": router f32) against the
// bf16 activations.  Selection is by logit, descending, with equal logits to the
// lower expert index (Trochilus, "What makes it different": the lowest row wins
// a tie).  Weights are the softmax over the k selected logits, which is the
// full softmax restricted to the selection and renormalised.
//
// Exactness.  f32 accumulation can reorder two experts whose logits are closer
// than its rounding error.  Each logit therefore carries a rigorous bound
//   |l_f32 - l_exact| <= beta = gamma_d * ||x_t||_2 * ||W_e||_2 (+ tiny terms)
// where d is the longest chain of roundings in the kernel's summation
// (gamma_d = d u / (1 - d u), u = 2^-24) and Cauchy-Schwarz bounds the sum of
// |x_h W_eh|.  A token whose selected set and selected order are separated by
// more than the bounds is certified; otherwise the candidates its bounds cannot
// rule out are recomputed in f64 from exact products (bf16 x f32 fits in 53
// bits) and selected again.  This is the "cheap bound first, exact work only
// where the bound reaches the best score" pattern of Trochilus's output head
// ("What makes it different").
#include "common.cuh"
#include "kernels.h"

namespace fp8moe {

// ------------------------------------------------------------------ logits, T small
// One CTA of 8 warps per expert row; warp w owns the column slice
// [w H/8, (w+1) H/8) and lane l the 4 columns 4 l + 128 j of that slice.  A
// lane sums its products sequentially with fma, a 5-level butterfly adds the
// 32 lanes, and one thread adds the 8 warp sums in order.  Rounding chain
// length: 4 ceil(H/1024) + 5 + 8 (+1 for the bias, added in the select
// kernel).  Also writes ||W_e||_2.
template <int TG>
__global__ void __launch_bounds__(256) router_logits_split_kernel(
    const __nv_bfloat16 *__restrict__ x, int64_t T, const float *__restrict__ W, int64_t E,
    int64_t H, float *__restrict__ logits, float *__restrict__ wnorm) {
  __shared__ float part[8][TG];
  __shared__ float ssq[8];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t e = blockIdx.x;
  const int64_t slice = H / 8;
  const int64_t h_lo = wid * slice, h_hi = h_lo + slice;
  const float *w = W + e * H;
  float ss = 0.f;
  for (int64_t h = h_lo + 4 * lane; h < h_hi; h += 128) {
    float4 wv = __ldg(reinterpret_cast<const float4 *>(w + h));
    ss = fmaf(wv.x, wv.x, ss);
    ss = fmaf(wv.y, wv.y, ss);
    ss = fmaf(wv.z, wv.z, ss);
    ss = fmaf(wv.w, wv.w, ss);
  }
  ss = warp_sum(ss);
  if (lane == 0) ssq[wid] = ss;

  for (int64_t t0 = 0; t0 < T; t0 += TG) {
    float acc[TG];
#pragma unroll
    for (int j = 0; j < TG; ++j) acc[j] = 0.f;
    for (int64_t h = h_lo + 4 * lane; h < h_hi; h += 128) {
      const float4 wv = __ldg(reinterpret_cast<const float4 *>(w + h));
#pragma unroll
      for (int j = 0; j < TG; ++j) {
        if (t0 + j < T) {
          const uint2 xv = __ldg(reinterpret_cast<const uint2 *>(x + (t0 + j) * H + h));
          acc[j] = fmaf(bf16_bits_to_float(xv.x & 0xffffu), wv.x, acc[j]);
          acc[j] = fmaf(bf16_bits_to_float(xv.x >> 16), wv.y, acc[j]);
          acc[j] = fmaf(bf16_bits_to_float(xv.y & 0xffffu), wv.z, acc[j]);
          acc[j] = fmaf(bf16_bits_to_float(xv.y >> 16), wv.w, acc[j]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < TG; ++j) {
      const float s = warp_sum(acc[j]);
      if (lane == 0) part[wid][j] = s;
    }
    __syncthreads();
    if (threadIdx.x < TG && t0 + threadIdx.x < T) {
      float v = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) v += part[q][threadIdx.x];
      logits[(t0 + threadIdx.x) * E + e] = v;
    }
    if (t0 == 0 && threadIdx.x == 32) {
      float v = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) v += ssq[q];
      wnorm[e] = sqrtf(v);
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ logits, T large
// Tiled SIMT product: a CTA computes 64 tokens x 64 experts, each thread a
// 4 x 4 block.  Each 128-wide K block is summed into a fresh partial by a
// chain of 128 fma, then added to the running total: rounding chain length
// 128 + H/128 (+1 for the bias).
__global__ void __launch_bounds__(256) router_logits_tiled_kernel(
    const __nv_bfloat16 *__restrict__ x, int64_t T, const float *__restrict__ W, int64_t E,
    int64_t H, float *__restrict__ logits) {
  // blockIdx.z selects a contiguous range of K blocks; its partial logits go
  // to plane z of logits [KS][T][E] and the select kernel adds the planes in
  // order (KS - 1 more roundings in the chain).
  const int64_t nkb_all = H / 128, ks = gridDim.z, z = blockIdx.z;
  const int64_t kb_lo = nkb_all * z / ks, kb_hi = nkb_all * (z + 1) / ks;
  logits += z * T * E;
  __shared__ __align__(16) float xs[32][68];
  __shared__ __align__(16) float ws[32][68];
  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int64_t t0 = (int64_t)blockIdx.y * 64, e0 = (int64_t)blockIdx.x * 64;
  float tot[4][4], part[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) tot[i][j] = 0.f;

  const int lr = tid >> 2;        // row of the tile this thread stages (0..63)
  const int lk = (tid & 3) * 8;   // first of its 8 k values
  for (int64_t kb = kb_lo * 128; kb < kb_hi * 128; kb += 128) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) part[i][j] = 0.f;
    for (int kt = 0; kt < 128; kt += 32) {
      const int64_t k0 = kb + kt + lk;
      {
        float v[8];
        if (t0 + lr < T) {
          uint4 xv = __ldg(reinterpret_cast<const uint4 *>(x + (t0 + lr) * H + k0));
          v[0] = bf16_bits_to_float(xv.x & 0xffffu); v[1] = bf16_bits_to_float(xv.x >> 16);
          v[2] = bf16_bits_to_float(xv.y & 0xffffu); v[3] = bf16_bits_to_float(xv.y >> 16);
          v[4] = bf16_bits_to_float(xv.z & 0xffffu); v[5] = bf16_bits_to_float(xv.z >> 16);
          v[6] = bf16_bits_to_float(xv.w & 0xffffu); v[7] = bf16_bits_to_float(xv.w >> 16);
        } else {
#pragma unroll
          for (int m = 0; m < 8; ++m) v[m] = 0.f;
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) xs[lk + m][lr] = v[m];
      }
      {
        float v[8];
        if (e0 + lr < E) {
          float4 a = __ldg(reinterpret_cast<const float4 *>(W + (e0 + lr) * H + k0));
          float4 b = __ldg(reinterpret_cast<const float4 *>(W + (e0 + lr) * H + k0 + 4));
          v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
#pragma unroll
          for (int m = 0; m < 8; ++m) v[m] = 0.f;
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) ws[lk + m][lr] = v[m];
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < 32; ++kk) {
        float4 a = *reinterpret_cast<const float4 *>(&xs[kk][ty * 4]);
        float4 b = *reinterpret_cast<const float4 *>(&ws[kk][tx * 4]);
        float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) part[i][j] = fmaf(av[i], bv[j], part[i][j]);
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) tot[i][j] += part[i][j];
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t e = e0 + tx * 4 + j;
      if (e < E) logits[t * E + e] = tot[i][j];
    }
  }
}

// ||W_e||_2, one warp per row.
__global__ void __launch_bounds__(128) row_norm_kernel(const float *__restrict__ W, int64_t E,
                                                       int64_t H, float *__restrict__ wnorm) {
  const int lane = threadIdx.x & 31;
  const int64_t e = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (e >= E) return;
  float ss = 0.f;
  for (int64_t h = 4 * lane; h < H; h += 128) {
    float4 wv = __ldg(reinterpret_cast<const float4 *>(W + e * H + h));
    ss = fmaf(wv.x, wv.x, ss);
    ss = fmaf(wv.y, wv.y, ss);
    ss = fmaf(wv.z, wv.z, ss);
    ss = fmaf(wv.w, wv.w, ss);
  }
  ss = warp_sum(ss);
  if (lane == 0) wnorm[e] = sqrtf(ss);
}

// ------------------------------------------------------------------ selection
// Argmax over the experts a lane owns (e = lane + 32 j) that are not yet taken,
// then over the warp: larger key first, lower expert on equal keys.
template <typename K, typename F>
__device__ __forceinline__ int warp_argmax(int E, uint32_t taken, F key, K *best_key) {
  const int lane = threadIdx.x & 31;
  K bk = K(0);
  int be = -1;
  for (int j = 0; lane + 32 * j < E; ++j) {
    if (taken >> j & 1u) continue;
    const int e = lane + 32 * j;
    const K v = key(e);
    if (be < 0 || v > bk) { bk = v; be = e; }  // ascending e: first max wins
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    K ok = __shfl_xor_sync(0xffffffffu, bk, o);
    int oe = __shfl_xor_sync(0xffffffffu, be, o);
    bool take = (oe >= 0) && (be < 0 || ok > bk || (ok == bk && oe < be));
    if (take) { bk = ok; be = oe; }
  }
  *best_key = bk;
  return be;
}

// One warp per token.  Shared memory per warp: E floats (logits + bias) and
// E doubles (refined logits).
__global__ void __launch_bounds__(128) router_select_kernel(
    const __nv_bfloat16 *__restrict__ x, int64_t T, const float *__restrict__ W,
    const float *__restrict__ bias, int64_t E, int64_t H, int k, const float *__restrict__ logits,
    const float *__restrict__ wnorm, int ks, float gamma_d, int32_t *__restrict__ idx,
    float *__restrict__ wts, __half *__restrict__ x16, float *__restrict__ xscale,
    int *__restrict__ err) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  const int64_t t = (int64_t)blockIdx.x * nw + wid;
  double *lg64 = reinterpret_cast<double *>(smem_raw) + (size_t)wid * E;
  float *lg = reinterpret_cast<float *>(smem_raw + (size_t)nw * E * sizeof(double)) + (size_t)wid * E;
  if (t >= T) return;
  const __nv_bfloat16 *xt = x + t * H;

  // ||x_t||_2 and max |x_t|
  float ss = 0.f, amax = 0.f;
  for (int64_t h = 4 * lane; h < H; h += 128) {
    uint2 xv = __ldg(reinterpret_cast<const uint2 *>(xt + h));
    float v0 = bf16_bits_to_float(xv.x & 0xffffu), v1 = bf16_bits_to_float(xv.x >> 16);
    float v2 = bf16_bits_to_float(xv.y & 0xffffu), v3 = bf16_bits_to_float(xv.y >> 16);
    ss = fmaf(v0, v0, ss); ss = fmaf(v1, v1, ss); ss = fmaf(v2, v2, ss); ss = fmaf(v3, v3, ss);
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3))));
  }
  const float xn = sqrtf(warp_sum(ss));
  amax = warp_max(amax);

  // f16 copy of x_t for the tensor-core GEMV, scaled by an exact power of two
  // so that the largest magnitude fits f16's range.
  if (x16 != nullptr) {
    const int sh = f16_range_shift(amax);
    const float down = exp2i(-sh);
    for (int64_t h = 4 * lane; h < H; h += 128) {
      uint2 xv = __ldg(reinterpret_cast<const uint2 *>(xt + h));
      uint2 o;
      o.x = pack_f16x2(bf16_bits_to_float(xv.x & 0xffffu) * down, bf16_bits_to_float(xv.x >> 16) * down);
      o.y = pack_f16x2(bf16_bits_to_float(xv.y & 0xffffu) * down, bf16_bits_to_float(xv.y >> 16) * down);
      *reinterpret_cast<uint2 *>(x16 + t * H + h) = o;
    }
    if (lane == 0) xscale[t] = exp2i(sh);
  }

  // f32 logits (+ bias) into shared memory
  bool finite = true;
  for (int e = lane; e < E; e += 32) {
    float v = logits[t * E + e];
    for (int z = 1; z < ks; ++z) v += logits[(z * T + t) * E + e];
    if (bias != nullptr) v += bias[e];
    finite = finite && isfinite(v);
    lg[e] = v;
  }
  if (!__all_sync(0xffffffffu, finite)) {
    if (lane == 0) set_error(err, DEV_ERR_NONFINITE);
    // still produce a valid routing: map non-finite logits to -inf below
  }
  __syncwarp();
  const float tiny = (float)H * 1.0e-37f;
  auto beta = [&](int e) -> float {
    float b = gamma_d * xn * wnorm[e] * 1.01f + tiny;
    if (bias != nullptr) b += fabsf(bias[e]) * 1.2e-7f;
    return b;
  };
  auto key32 = [&](int e) -> float {
    float v = lg[e];
    return isfinite(v) ? v : -INFINITY;
  };

  // f32 selection of the top k
  uint32_t taken = 0;
  int sel_e = -1;      // lane r holds the expert of rank r
  float sel_v = 0.f;
  for (int r = 0; r < k; ++r) {
    float bv;
    int be = warp_argmax<float>((int)E, taken, key32, &bv);
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == r) { sel_e = be; sel_v = bv; }
  }
  // certify: every selected lower bound above every other upper bound, and
  // adjacent selected experts separated by their bounds
  float upper_rest = -INFINITY;
  for (int j = 0; lane + 32 * j < E; ++j) {
    if (taken >> j & 1u) continue;
    const int e = lane + 32 * j;
    upper_rest = fmaxf(upper_rest, key32(e) + beta(e));
  }
  upper_rest = warp_max(upper_rest);
  float lo_sel = (lane < k) ? sel_v - beta(sel_e) : INFINITY;
  float hi_next = __shfl_down_sync(0xffffffffu, (lane < k) ? sel_v + beta(sel_e) : -INFINITY, 1);
  bool ordered = (lane + 1 >= k) || (lo_sel > hi_next);
  float min_lo = -warp_max(-lo_sel);
  bool certified = __all_sync(0xffffffffu, ordered) && (k == E || min_lo > upper_rest) &&
                   isfinite(min_lo);

  if (certified) {
    const float l0 = __shfl_sync(0xffffffffu, sel_v, 0);
    float ex = (lane < k) ? __expf(sel_v - l0) : 0.f;
    float z = warp_sum(ex);
    if (lane < k) {
      idx[t * k + lane] = sel_e;
      wts[t * k + lane] = ex / z;
    }
    return;
  }

  // Refinement: the k-th largest lower bound; every expert whose upper bound
  // reaches it is a candidate and is recomputed in f64.
  uint32_t taken2 = 0;
  float kth_lo = -INFINITY;
  auto lo_key = [&](int e) -> float { return key32(e) - beta(e); };
  for (int r = 0; r < k; ++r) {
    float bv;
    int be = warp_argmax<float>((int)E, taken2, lo_key, &bv);
    if ((be & 31) == lane) taken2 |= 1u << (be >> 5);
    kth_lo = bv;
  }
  // candidates: each lane tests its own experts; the warp then recomputes
  // them one at a time (lane order, then j), all lanes cooperating on the dot
  uint32_t cmask = 0;
  for (int j = 0; lane + 32 * j < E; ++j) {
    const int e = lane + 32 * j;
    if (!(key32(e) + beta(e) < kth_lo) && isfinite(lg[e])) cmask |= 1u << j;
    else lg64[e] = -INFINITY;
  }
  for (int src = 0; src < 32; ++src) {
    uint32_t m = __shfl_sync(0xffffffffu, cmask, src);
    while (m != 0u) {
      const int j = __ffs(m) - 1;
      m &= m - 1u;
      const int e = src + 32 * j;
      const float *w = W + (int64_t)e * H;
      double acc = 0.0;
      for (int64_t h = 4 * lane; h < H; h += 128) {
        float4 wv = __ldg(reinterpret_cast<const float4 *>(w + h));
        uint2 xv = __ldg(reinterpret_cast<const uint2 *>(xt + h));
        acc = fma((double)bf16_bits_to_float(xv.x & 0xffffu), (double)wv.x, acc);
        acc = fma((double)bf16_bits_to_float(xv.x >> 16), (double)wv.y, acc);
        acc = fma((double)bf16_bits_to_float(xv.y & 0xffffu), (double)wv.z, acc);
        acc = fma((double)bf16_bits_to_float(xv.y >> 16), (double)wv.w, acc);
      }
      double v = warp_sum(acc);
      if (bias != nullptr) v += (double)bias[e];
      if (lane == 0) lg64[e] = v;
    }
  }
  __syncwarp();
  auto key64 = [&](int e) -> double { return lg64[e]; };
  uint32_t taken3 = 0;
  int fe = -1;
  double fv = 0.0;
  for (int r = 0; r < k; ++r) {
    double bv;
    int be = warp_argmax<double>((int)E, taken3, key64, &bv);
    if ((be & 31) == lane) taken3 |= 1u << (be >> 5);
    if (lane == r) { fe = be; fv = bv; }
  }
  const double l0 = __shfl_sync(0xffffffffu, fv, 0);
  double ex = (lane < k) ? exp(fv - l0) : 0.0;
  double z = warp_sum(ex);
  if (lane < k) {
    if (fe < 0 || fe >= E) { set_error(err, DEV_ERR_BOUNDS); fe = 0; }
    idx[t * k + lane] = fe;
    wts[t * k + lane] = (float)(ex / z);
  }
}

// ------------------------------------------------------------------ launchers

int router_k_split(int64_t T, int64_t E, int64_t H, int sms) {
  if (T <= kRouterWarpMaxT) return 1;
  const int64_t tiles = ((T + 63) / 64) * ((E + 63) / 64);
  int64_t ks = (2 * sms + tiles - 1) / tiles;
  const int64_t nkb = H / 128;
  if (ks > nkb) ks = nkb;
  if (ks > kRouterMaxKSplit) ks = kRouterMaxKSplit;
  return ks < 1 ? 1 : (int)ks;
}

int router_chain_depth(int64_t T, int64_t H, int ks) {
  return T <= kRouterWarpMaxT ? (int)(4 * ((H + 1023) / 1024) + 5 + 8 + 1)
                              : (int)(128 + H / 128 + ks + 1);
}

cudaError_t launch_router_logits(const __nv_bfloat16 *x, int64_t T, const float *W, int64_t E,
                                 int64_t H, int ks, float *logits, float *wnorm, cudaStream_t s) {
  if (T <= kRouterWarpMaxT) {
    if (T <= 1)
      router_logits_split_kernel<1><<<(unsigned)E, 256, 0, s>>>(x, T, W, E, H, logits, wnorm);
    else
      router_logits_split_kernel<8><<<(unsigned)E, 256, 0, s>>>(x, T, W, E, H, logits, wnorm);
    return cudaGetLastError();
  }
  row_norm_kernel<<<(unsigned)((E + 3) / 4), 128, 0, s>>>(W, E, H, wnorm);
  dim3 grid((unsigned)((E + 63) / 64), (unsigned)((T + 63) / 64), (unsigned)ks);
  router_logits_tiled_kernel<<<grid, 256, 0, s>>>(x, T, W, E, H, logits);
  return cudaGetLastError();
}

size_t router_select_smem(int64_t E) { return (size_t)4 * E * (sizeof(double) + sizeof(float)); }

cudaError_t launch_router_select(const __nv_bfloat16 *x, int64_t T, const float *W,
                                 const float *bias, int64_t E, int64_t H, int k,
                                 const float *logits, const float *wnorm, int ks, float gamma_d,
                                 int32_t *idx, float *wts, __half *x16, float *xscale, int *err,
                                 cudaStream_t s) {
  const size_t smem = router_select_smem(E);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(router_select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  router_select_kernel<<<(unsigned)((T + 3) / 4), 128, smem, s>>>(
      x, T, W, bias, E, H, k, logits, wnorm, ks, gamma_d, idx, wts, x16, xscale, err);
  return cudaGetLastError();
}

}  // namespace fp8moe
