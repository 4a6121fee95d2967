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
// rule out are recomputed from exact products, with every rounding error
// carried (exact_logit), and selected again.  This is the "cheap bound first, exact work only
// where the bound reaches the best score" pattern of Trochilus's output head
// ("What makes it different").
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "permute.cuh"

namespace fp8moe {

// ------------------------------------------------------------------ selection
struct SelectArgs {
  const __nv_bfloat16 *x;
  int64_t T;
  const float *W, *bias;
  int64_t E, H;
  int k;
  const float *logits;  // ks planes [ks][T][E] of partial logits
  int ks;
  const float *wnorm;   // ||W_e||_2
  float gamma;          // gamma_d of the logit kernel's rounding chain
  int32_t *idx;
  float *wts;
  int *err;
};

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

// ||x_t||_2 and max |x_t| by one warp (4 independent partial sums per lane
// keep several loads in flight).
__device__ __forceinline__ void x_stats(const __nv_bfloat16 *xt, int64_t H, float *norm, float *amax) {
  const int lane = threadIdx.x & 31;
  float ss = 0.f, am = 0.f;
#pragma unroll 4
  for (int64_t h = 4 * lane; h < H; h += 128) {
    const uint2 xv = __ldg(reinterpret_cast<const uint2 *>(xt + h));
    const float v0 = bf16_bits_to_float(xv.x & 0xffffu), v1 = bf16_bits_to_float(xv.x >> 16);
    const float v2 = bf16_bits_to_float(xv.y & 0xffffu), v3 = bf16_bits_to_float(xv.y >> 16);
    ss = fmaf(v0, v0, ss); ss = fmaf(v1, v1, ss); ss = fmaf(v2, v2, ss); ss = fmaf(v3, v3, ss);
    am = fmaxf(am, fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3))));
  }
  *norm = sqrtf(warp_sum(ss));
  *amax = warp_max(am);
}

// f16 copy of x_t for the tensor-core GEMV, scaled by an exact power of two
// so that the largest magnitude fits f16's range; xscale[t] undoes it.
__device__ __forceinline__ void x_to_f16(const __nv_bfloat16 *xt, int64_t H, float amax,
                                         __half *x16t, float *xscale_t) {
  const int lane = threadIdx.x & 31;
  const int sh = f16_range_shift(amax);
  const float down = exp2i(-sh);
#pragma unroll 4
  for (int64_t h = 4 * lane; h < H; h += 128) {
    const uint2 xv = __ldg(reinterpret_cast<const uint2 *>(xt + h));
    uint2 o;
    o.x = pack_f16x2(bf16_bits_to_float(xv.x & 0xffffu) * down, bf16_bits_to_float(xv.x >> 16) * down);
    o.y = pack_f16x2(bf16_bits_to_float(xv.y & 0xffffu) * down, bf16_bits_to_float(xv.y >> 16) * down);
    *reinterpret_cast<uint2 *>(x16t + h) = o;
  }
  if (lane == 0) *xscale_t = exp2i(sh);
}

// Error-free f32 steps for the exact logits: x * w = p + q exactly (p the
// rounded product, q = fma(x, w, -p)), and a + b = s + err exactly (Knuth's
// TwoSum).  The _rn intrinsics keep the compiler from contracting or
// reordering them.
__device__ __forceinline__ void two_prod(float x, float w, float &p, float &q) {
  p = __fmul_rn(x, w);
  q = fmaf(x, w, -p);
}
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &err) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
// Adds x * w into the unevaluated sum hi + lo.
__device__ __forceinline__ void acc_exact(float x, float w, float &hi, float &lo) {
  float p, q, s, e;
  two_prod(x, w, p, q);
  two_sum(hi, p, s, e);
  hi = s;
  lo = __fadd_rn(lo, __fadd_rn(e, q));
}

// logit of expert e for x_t, by the whole warp, from exact products: every
// product and every addition's rounding error is carried in f32 pairs (hi +
// lo, eight independent chains per lane), whose sum in f64 differs from the
// exact dot product by at most about n^2 2^-48 of sum |x W| (n = H / 256
// products per chain: 2e-12 of it at H = 6144, 3.7e-12 at H = 8192).  The
// f32 pipes are many times wider than the f64 one; eight loads per lane are
// in flight.
__device__ __forceinline__ double exact_logit(const SelectArgs &a, const __nv_bfloat16 *xt, int e) {
  const int lane = threadIdx.x & 31;
  const float *w = a.W + (int64_t)e * a.H;
  constexpr int U = 8;  // loads per lane in flight (chains)
  float hi[U], lo[U];
#pragma unroll
  for (int u = 0; u < U; ++u) hi[u] = lo[u] = 0.f;
  for (int64_t h0 = 4 * lane; h0 < a.H; h0 += 128 * U) {
    float4 wv[U];
    uint2 xv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t h = h0 + 128 * u;
      wv[u] = h < a.H ? __ldg(reinterpret_cast<const float4 *>(w + h)) : make_float4(0.f, 0.f, 0.f, 0.f);
      xv[u] = h < a.H ? __ldg(reinterpret_cast<const uint2 *>(xt + h)) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      acc_exact(bf16_bits_to_float(xv[u].x & 0xffffu), wv[u].x, hi[u], lo[u]);
      acc_exact(bf16_bits_to_float(xv[u].x >> 16), wv[u].y, hi[u], lo[u]);
      acc_exact(bf16_bits_to_float(xv[u].y & 0xffffu), wv[u].z, hi[u], lo[u]);
      acc_exact(bf16_bits_to_float(xv[u].y >> 16), wv[u].w, hi[u], lo[u]);
    }
  }
  double acc[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) acc[u] = ((double)hi[u] + (double)lo[u]) + ((double)hi[u + 4] + (double)lo[u + 4]);
  double v = warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
  if (a.bias != nullptr) v += (double)a.bias[e];
  return v;
}

// Top-k of token t by one warp.  Per-warp shared memory: lg and bt (E floats
// each: logits + bias and their error bounds) and lg64 (E doubles).  Logits
// are read with ld.global.cg so that planes written by other CTAs of the same
// grid are seen.  Kept out of line: the small-batch selection calls it only
// for tokens its bound cannot certify, and a launch that follows an L2 flush
// pays for every instruction line it fetches, so this code stays off that
// kernel's common path.
__device__ __noinline__ void select_token(const SelectArgs &a, int64_t t, float xn, float *lg, float *bt,
                             double *lg64) {
  const int lane = threadIdx.x & 31;
  const int E = (int)a.E, k = a.k;
  const __nv_bfloat16 *xt = a.x + t * a.H;

  const float tiny = (float)a.H * 1.0e-37f;
  bool finite = true;
#pragma unroll 4
  for (int e = lane; e < E; e += 32) {
    float v = __ldcg(a.logits + t * a.E + e);
    for (int z = 1; z < a.ks; ++z) v += __ldcg(a.logits + (z * a.T + t) * a.E + e);
    float b = a.gamma * xn * __ldcg(a.wnorm + e) * 1.01f + tiny;
    if (a.bias != nullptr) {
      const float bb = a.bias[e];
      v += bb;
      b += fabsf(bb) * 1.2e-7f;
    }
    finite = finite && isfinite(v);
    lg[e] = v;
    bt[e] = b;
  }
  if (!__all_sync(0xffffffffu, finite) && lane == 0) set_error(a.err, DEV_ERR_NONFINITE);
  __syncwarp();
  auto beta = [&](int e) -> float { return bt[e]; };
  auto key32 = [&](int e) -> float {
    const float v = lg[e];
    return isfinite(v) ? v : -INFINITY;
  };

  // f32 selection of the top k
  uint32_t taken = 0;
  int sel_e = -1;  // lane r holds the expert of rank r
  float sel_v = 0.f;
  for (int r = 0; r < k; ++r) {
    float bv;
    const int be = warp_argmax<float>(E, taken, key32, &bv);
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
  const float lo_sel = (lane < k) ? sel_v - beta(sel_e) : INFINITY;
  const float hi_next = __shfl_down_sync(0xffffffffu, (lane < k) ? sel_v + beta(sel_e) : -INFINITY, 1);
  const bool ordered = (lane + 1 >= k) || (lo_sel > hi_next);
  const float min_lo = -warp_max(-lo_sel);
  const bool certified = __all_sync(0xffffffffu, ordered) && (k == E || min_lo > upper_rest) &&
                         isfinite(min_lo);

  if (certified) {
    const float l0 = __shfl_sync(0xffffffffu, sel_v, 0);
    const float ex = (lane < k) ? __expf(sel_v - l0) : 0.f;
    const float z = warp_sum(ex);
    if (lane < k) {
      a.idx[t * k + lane] = sel_e;
      a.wts[t * k + lane] = ex / z;
    }
    return;
  }

  // Refinement.  Candidates: every expert whose upper bound reaches the k-th
  // largest lower bound (the others are certainly below k experts).  A
  // candidate whose interval [l - beta, l + beta] overlaps no other
  // candidate's is "isolated": its f32 value already orders it correctly
  // against every candidate.  Only the others are recomputed from exact
  // products (exact_logit); the top k is then taken on key = recomputed value
  // or f32 value (isolated), which orders every pair of candidates exactly.
  uint32_t taken2 = 0;
  float kth_lo = -INFINITY;
  auto lo_key = [&](int e) -> float { return key32(e) - beta(e); };
  for (int r = 0; r < k; ++r) {
    float bv;
    const int be = warp_argmax<float>(E, taken2, lo_key, &bv);
    if ((be & 31) == lane) taken2 |= 1u << (be >> 5);
    kth_lo = bv;
  }
  uint32_t cmask = 0;
  for (int j = 0; lane + 32 * j < E; ++j) {
    const int e = lane + 32 * j;
    if (!(key32(e) + beta(e) < kth_lo) && isfinite(lg[e])) cmask |= 1u << j;
  }
  // compact the candidates to one per lane (at most 32; more only in
  // degenerate near-total ties, where every candidate is recomputed)
  const int ccount = __popc(cmask);
  int cpre = ccount;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, cpre, o);
    if (lane >= o) cpre += n;
  }
  const int ctotal = __shfl_sync(0xffffffffu, cpre, 31);
  cpre -= ccount;
  int *cand = reinterpret_cast<int *>(lg64);  // first 32 slots; lg64 is rewritten below
  const bool compact = ctotal <= 32;
  double key = -INFINITY;
  int my_e = -1;
  if (compact) {
    {
      uint32_t m = cmask;
      int slot = cpre;
      while (m != 0u) {
        const int j = __ffs(m) - 1;
        m &= m - 1u;
        cand[slot++] = lane + 32 * j;
      }
    }
    __syncwarp();
    my_e = lane < ctotal ? cand[lane] : -1;
    __syncwarp();
    const float mv = my_e >= 0 ? lg[my_e] : 0.f, mb = my_e >= 0 ? bt[my_e] : 0.f;
    const float mlo = mv - mb, mup = mv + mb;
    bool isolated = true;
    for (int s2 = 0; s2 < ctotal; ++s2) {
      const float olo = __shfl_sync(0xffffffffu, mlo, s2), oup = __shfl_sync(0xffffffffu, mup, s2);
      if (s2 != lane && mlo <= oup && olo <= mup) isolated = false;
    }
    uint32_t rmask = __ballot_sync(0xffffffffu, my_e >= 0 && !isolated);
    key = my_e >= 0 ? (double)mv : -INFINITY;
    while (rmask != 0u) {
      const int src = __ffs(rmask) - 1;
      rmask &= rmask - 1u;
      const int e = __shfl_sync(0xffffffffu, my_e, src);
      const double v = exact_logit(a, xt, e);
      if (lane == src) key = v;
    }
  } else {
    for (int j = 0; lane + 32 * j < E; ++j) lg64[lane + 32 * j] = -INFINITY;
    __syncwarp();
    for (int src = 0; src < 32; ++src) {
      uint32_t m = __shfl_sync(0xffffffffu, cmask, src);
      while (m != 0u) {
        const int j = __ffs(m) - 1;
        m &= m - 1u;
        const int e = src + 32 * j;
        const double v = exact_logit(a, xt, e);
        if (lane == 0) lg64[e] = v;
      }
    }
    __syncwarp();
  }

  // top k on the keys, larger first, lower expert on equal keys
  int fe = -1;
  double fv = 0.0;
  if (compact) {
    bool used = my_e < 0;
    for (int r = 0; r < k; ++r) {
      double bk = used ? -INFINITY : key;
      int be = used ? INT_MAX : my_e;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const double ok = __shfl_xor_sync(0xffffffffu, bk, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ok > bk || (ok == bk && oe < be)) { bk = ok; be = oe; }
      }
      if (be == my_e) used = true;
      if (lane == r) { fe = be; fv = bk; }
    }
  } else {
    auto key64 = [&](int e) -> double { return lg64[e]; };
    uint32_t taken3 = 0;
    for (int r = 0; r < k; ++r) {
      double bv;
      const int be = warp_argmax<double>(E, taken3, key64, &bv);
      if ((be & 31) == lane) taken3 |= 1u << (be >> 5);
      if (lane == r) { fe = be; fv = bv; }
    }
  }
  const double l0 = __shfl_sync(0xffffffffu, fv, 0);
  const double ex = (lane < k) ? exp(fv - l0) : 0.0;
  const double z = warp_sum(ex);
  if (lane < k) {
    if (fe < 0 || fe >= E) { set_error(a.err, DEV_ERR_BOUNDS); fe = 0; }
    a.idx[t * k + lane] = fe;
    a.wts[t * k + lane] = (float)(ex / z);
  }
}

// ------------------------------------------------------------------ fused small-batch routing
// One launch for T <= 64.  CTA e computes the logits of expert e for every
// token (8 warps split H: lane chain 4 ceil(H/1024), butterfly 5, warp sum 8,
// +1 bias) and ||W_e||; the same pass gives every CTA ||x_t|| and max |x_t|,
// and CTA c % E writes 128-column chunk c of the f16 copy of x.  The last CTA
// to finish (an atomic ticket, reset for the next call) selects the top k of
// every token and sorts the pairs by expert.
constexpr int kRouteWarps = 8;

template <int TG>
__global__ void __launch_bounds__(32 * kRouteWarps) route_decode_kernel(
    SelectArgs a, float *__restrict__ logits_w, float *__restrict__ wnorm_w,
    float *__restrict__ xnorm, __half *__restrict__ x16, float *__restrict__ xscale,
    int32_t *__restrict__ ticket, int tile_m, SortOut so, uint32_t *__restrict__ pos_max) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ float part[kRouteWarps][TG], part_ss[kRouteWarps][TG], part_am[kRouteWarps][TG];
  __shared__ float ssq[kRouteWarps];
  __shared__ float s_am[kRouterWarpMaxT];
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t E = a.E, H = a.H, T = a.T;
  const int64_t e = blockIdx.x;
  pdl_trigger();  // the next kernel may be scheduled; it waits for this one to finish

  // ---- phase A: logits of expert e, ||W_e||, and (redundantly in every CTA,
  // from the same pass over x) ||x_t|| and max |x_t|
  const int64_t slice = H / kRouteWarps;
  const int64_t h_lo = wid * slice, h_hi = h_lo + slice;
  const float *w = a.W + e * H;
  float ss = 0.f;
  for (int64_t hh = h_lo + 4 * lane; hh < h_hi; hh += 128) {
    const float4 wv = __ldg(reinterpret_cast<const float4 *>(w + hh));
    ss = fmaf(wv.x, wv.x, ss);
    ss = fmaf(wv.y, wv.y, ss);
    ss = fmaf(wv.z, wv.z, ss);
    ss = fmaf(wv.w, wv.w, ss);
  }
  ss = warp_sum(ss);
  if (lane == 0) ssq[wid] = ss;
  for (int64_t t0 = 0; t0 < T; t0 += TG) {
    float acc[TG], xs[TG], xm[TG];
#pragma unroll
    for (int j = 0; j < TG; ++j) { acc[j] = 0.f; xs[j] = 0.f; xm[j] = 0.f; }
    for (int64_t hh = h_lo + 4 * lane; hh < h_hi; hh += 128) {
      const float4 wv = __ldg(reinterpret_cast<const float4 *>(w + hh));
#pragma unroll
      for (int j = 0; j < TG; ++j) {
        if (t0 + j < T) {
          const uint2 xv = __ldg(reinterpret_cast<const uint2 *>(a.x + (t0 + j) * H + hh));
          const float v0 = bf16_bits_to_float(xv.x & 0xffffu), v1 = bf16_bits_to_float(xv.x >> 16);
          const float v2 = bf16_bits_to_float(xv.y & 0xffffu), v3 = bf16_bits_to_float(xv.y >> 16);
          acc[j] = fmaf(v0, wv.x, acc[j]);
          acc[j] = fmaf(v1, wv.y, acc[j]);
          acc[j] = fmaf(v2, wv.z, acc[j]);
          acc[j] = fmaf(v3, wv.w, acc[j]);
          xs[j] = fmaf(v0, v0, xs[j]); xs[j] = fmaf(v1, v1, xs[j]);
          xs[j] = fmaf(v2, v2, xs[j]); xs[j] = fmaf(v3, v3, xs[j]);
          xm[j] = fmaxf(xm[j], fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3))));
        }
      }
    }
#pragma unroll
    for (int j = 0; j < TG; ++j) {
      const float s = warp_sum(acc[j]), q2 = warp_sum(xs[j]), m = warp_max(xm[j]);
      if (lane == 0) { part[wid][j] = s; part_ss[wid][j] = q2; part_am[wid][j] = m; }
    }
    __syncthreads();
    if (threadIdx.x < TG && t0 + threadIdx.x < T) {
      float v = 0.f, q2 = 0.f, m = 0.f;
#pragma unroll
      for (int q = 0; q < kRouteWarps; ++q) {
        v += part[q][threadIdx.x];
        q2 += part_ss[q][threadIdx.x];
        m = fmaxf(m, part_am[q][threadIdx.x]);
      }
      const int64_t t = t0 + threadIdx.x;
      logits_w[t * E + e] = v;
      s_am[t] = m;
      if (e == 0) {
        xnorm[t] = sqrtf(q2);
        if (xscale != nullptr) xscale[t] = exp2i(f16_range_shift(m));
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 32) {
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < kRouteWarps; ++q) v += ssq[q];
    wnorm_w[e] = sqrtf(v);
  }
  // f16 copy of x: 128-column chunk c of every token is written by CTA c % E,
  // scaled by the token's exact power of two (max |x_t| known from the pass)
  if (x16 != nullptr) {
    const int64_t nch = H / 128;
    for (int64_t c = e; c < nch; c += E) {
      for (int64_t t = wid; t < T; t += kRouteWarps) {
        const float down = exp2i(-f16_range_shift(s_am[t]));
        const int64_t h = c * 128 + 4 * lane;
        const uint2 xv = __ldg(reinterpret_cast<const uint2 *>(a.x + t * H + h));
        uint2 o;
        o.x = pack_f16x2(bf16_bits_to_float(xv.x & 0xffffu) * down, bf16_bits_to_float(xv.x >> 16) * down);
        o.y = pack_f16x2(bf16_bits_to_float(xv.y & 0xffffu) * down, bf16_bits_to_float(xv.y >> 16) * down);
        *reinterpret_cast<uint2 *>(x16 + t * H + h) = o;
      }
    }
  }

  // ---- ticket: the last CTA continues
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(ticket, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // ---- phase B: selection (warp per token), then the stable sort
  double *lg64 = reinterpret_cast<double *>(smem_raw) + (size_t)wid * E;
  float *lg = reinterpret_cast<float *>(smem_raw + (size_t)kRouteWarps * E * sizeof(double)) + (size_t)wid * 2 * E;
  for (int64_t t = wid; t < T; t += kRouteWarps) select_token(a, t, __ldcg(xnorm + t), lg, lg + E, lg64);
  if (pos_max != nullptr)
    for (int64_t p = threadIdx.x; p < T * a.k; p += blockDim.x) pos_max[p] = 0u;
  __threadfence_block();
  __syncthreads();
  cta_counting_sort<kRouteWarps>(a.idx, T * a.k, (int)E, tile_m, so, reinterpret_cast<int *>(smem_raw), a.err);
  if (threadIdx.x == 0) *ticket = 0;
}

// ------------------------------------------------------------------ small-batch routing
// T <= 64 on the tensor-core decode path, in two launches chained by
// programmatic dependent launch.
//
// Logits: the grid is (expert blocks) x (token blocks of 8).  CTA (eb, tb)
// computes the logits of EPC experts for the tb's tokens: WPE = 8 / EPC warps
// share one expert's row, each over a contiguous range of 128-column chunks
// (four chunks' loads in flight at a time); a lane keeps four partial sums
// (one per column of its 4-column slice), so the longest rounding chain is
// nch_w + 2 (lane) + 5 (butterfly) + log2(WPE) (pairwise over warps) + 1
// (bias), nch_w = ceil(H / 128 / WPE).  The same CTAs split every token row of
// the block into per-(token, 128-column chunk) units: two e4m3 terms with one
// power-of-two scale (the tensor-core FFN's activation operand, token-major)
// and the chunk's sum of squares (for ||x_t||).
//
// Selection and sort: one CTA.  Each warp takes tokens t = warp, warp + NW,
// ..: it holds the token's logits and bounds in registers (EPL per lane),
// selects the top k and certifies the order as the general selection does;
// a token the bound cannot certify goes through the exact path
// (select_token).  Warp 0 then sorts the pairs by expert from shared memory
// while the other warps clear the FFN's work counters.
constexpr int kSmallTB = 8;  // tokens per token block

struct RouteSmallArgs {
  SelectArgs sel;             // logits [T][E], wnorm [E], idx, wts, err
  int epc;                    // experts per CTA (1, 2, 4 or 8)
  float *logits_w, *wnorm_w;
  float *xss;                 // [T][H/128] per-chunk sums of squares
  uint8_t *a_hi, *a_lo;       // [T, H] activation terms (token-major)
  float *a_scale;             // [H/128][a_ld] power-of-two scales
  int64_t a_ld;
  int32_t *counters;          // [n_counters] cleared for the expert kernels
  int n_counters;
  int tile_m;
  SortOut so;
};

__global__ void __launch_bounds__(32 * kRouteWarps) route_logits_small_kernel(RouteSmallArgs r) {
  __shared__ float part_l[kRouteWarps][kSmallTB];
  __shared__ float part_w[kRouteWarps];
  const SelectArgs &a = r.sel;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t E = a.E, H = a.H, T = a.T;
  const int64_t nch = H / 128;
  const int epc = r.epc, wpe = kRouteWarps / epc;
  const int eb = blockIdx.x, tb = blockIdx.y, n_eb = gridDim.x;
  const int64_t t0 = (int64_t)tb * kSmallTB;
  const int nt = (int)((T - t0) < kSmallTB ? (T - t0) : kSmallTB);
  pdl_trigger();  // the selection kernel may be scheduled; it waits for this grid

  // ---- logits of EPC experts for the block's tokens
  const int eslot = wid / wpe, part = wid % wpe;
  const int64_t e = (int64_t)eb * epc + eslot;
  const int64_t c_lo = nch * part / wpe, c_hi = nch * (part + 1) / wpe;
  float acc[kSmallTB][4], wss[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < kSmallTB; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;
  if (e < E) {
    const float *w = a.W + e * H;
    for (int64_t c0 = c_lo; c0 < c_hi; c0 += 4) {
      // four chunks' loads in flight, then their products
      float4 wv[4];
      uint2 xv[4][kSmallTB];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t h = (c0 + u) * 128 + 4 * lane;
        const bool in = c0 + u < c_hi;
        wv[u] = in ? __ldg(reinterpret_cast<const float4 *>(w + h)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < kSmallTB; ++j)
          xv[u][j] = (in && j < nt) ? __ldg(reinterpret_cast<const uint2 *>(a.x + (t0 + j) * H + h))
                                    : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        wss[0] = fmaf(wv[u].x, wv[u].x, wss[0]);
        wss[1] = fmaf(wv[u].y, wv[u].y, wss[1]);
        wss[2] = fmaf(wv[u].z, wv[u].z, wss[2]);
        wss[3] = fmaf(wv[u].w, wv[u].w, wss[3]);
#pragma unroll
        for (int j = 0; j < kSmallTB; ++j) {
          acc[j][0] = fmaf(bf16_bits_to_float(xv[u][j].x & 0xffffu), wv[u].x, acc[j][0]);
          acc[j][1] = fmaf(bf16_bits_to_float(xv[u][j].x >> 16), wv[u].y, acc[j][1]);
          acc[j][2] = fmaf(bf16_bits_to_float(xv[u][j].y & 0xffffu), wv[u].z, acc[j][2]);
          acc[j][3] = fmaf(bf16_bits_to_float(xv[u][j].y >> 16), wv[u].w, acc[j][3]);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kSmallTB; ++j) {
    const float v = warp_sum((acc[j][0] + acc[j][1]) + (acc[j][2] + acc[j][3]));
    if (lane == 0) part_l[wid][j] = v;
  }
  {
    const float v = warp_sum((wss[0] + wss[1]) + (wss[2] + wss[3]));
    if (lane == 0) part_w[wid] = v;
  }

  // ---- activation units (token j of the block, chunk c), split over the
  // warps of the token block's CTAs
  {
    const int64_t n_units = (int64_t)nt * nch;
    for (int64_t u = (int64_t)eb * kRouteWarps + wid; u < n_units; u += (int64_t)n_eb * kRouteWarps) {
      const int64_t t = t0 + u / nch, c = u % nch;
      const int64_t col = c * 128 + 4 * lane;
      const uint2 xv = __ldg(reinterpret_cast<const uint2 *>(a.x + t * H + col));
      const float v0 = bf16_bits_to_float(xv.x & 0xffffu), v1 = bf16_bits_to_float(xv.x >> 16);
      const float v2 = bf16_bits_to_float(xv.y & 0xffffu), v3 = bf16_bits_to_float(xv.y >> 16);
      const float am = warp_max(fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3))));
      const float ss = warp_sum((v0 * v0 + v1 * v1) + (v2 * v2 + v3 * v3));
      const int ex = e4m3_block_exponent(am);
      const Pow2 down = pow2_factors(-ex);
      uint32_t p[2], q[2];
      e4m3_terms<2>(down(v0), down(v1), p);
      e4m3_terms<2>(down(v2), down(v3), q);
      *reinterpret_cast<uint32_t *>(r.a_hi + t * H + col) = p[0] | (q[0] << 16);
      *reinterpret_cast<uint32_t *>(r.a_lo + t * H + col) = p[1] | (q[1] << 16);
      if (lane == 0) {
        r.a_scale[c * r.a_ld + t] = ldexpf(1.f, ex);
        r.xss[t * nch + c] = ss;
      }
    }
  }
  __syncthreads();
  // pairwise tree over the WPE warps of an expert, in a fixed order
  if (threadIdx.x < epc * kSmallTB) {
    const int es = threadIdx.x / kSmallTB, j = threadIdx.x % kSmallTB;
    const int64_t ee = (int64_t)eb * epc + es;
    float v[kRouteWarps];
#pragma unroll
    for (int q = 0; q < kRouteWarps; ++q) v[q] = q < wpe ? part_l[es * wpe + q][j] : 0.f;
    for (int w = 1; w < wpe; w <<= 1)
      for (int q = 0; q + w < wpe; q += 2 * w) v[q] = v[q] + v[q + w];
    if (ee < E && j < nt) r.logits_w[(t0 + j) * E + ee] = v[0];
    if (ee < E && j == 0 && tb == 0) {
      float ssum = 0.f;
      for (int q = 0; q < wpe; ++q) ssum += part_w[es * wpe + q];
      r.wnorm_w[ee] = sqrtf(ssum);
    }
  }
}

// Top k of token t from register-held logits (EPL per lane, expert
// lane + 32 i); the same selection, certification and weights as
// select_token's certified case.  Returns false (writing nothing) when the
// bound cannot certify the order or a logit is not finite; the caller then
// runs the exact path.
template <int EPL>
__device__ bool select_fast(const SelectArgs &a, int64_t t, float xn, int32_t *idx_s) {
  const int lane = threadIdx.x & 31;
  const int E = (int)a.E, k = a.k;
  const float tiny = (float)a.H * 1.0e-37f;
  float v[EPL], b[EPL];
  bool finite = true;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      float lv = __ldcg(a.logits + t * a.E + e);
      float bb = a.gamma * xn * __ldcg(a.wnorm + e) * 1.01f + tiny;
      if (a.bias != nullptr) {
        const float bi = __ldg(a.bias + e);
        lv += bi;
        bb += fabsf(bi) * 1.2e-7f;
      }
      finite = finite && isfinite(lv);
      v[i] = lv;
      b[i] = bb;
    } else {
      v[i] = -INFINITY;
      b[i] = 0.f;
    }
  }
  if (!__all_sync(0xffffffffu, finite)) return false;
  uint32_t taken = 0;
  int sel_e = -1;
  float sel_v = 0.f, sel_b = 0.f;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY, bb = 0.f;
    int be = INT_MAX;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (!((taken >> i) & 1u) && e < E && (be == INT_MAX || v[i] > bv)) {
        bv = v[i];
        be = e;
        bb = b[i];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      const float ob = __shfl_xor_sync(0xffffffffu, bb, o);
      if (oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be))) {
        bv = ov;
        be = oe;
        bb = ob;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == r) {
      sel_e = be;
      sel_v = bv;
      sel_b = bb;
    }
  }
  // certify: every selected lower bound above every other upper bound, and
  // adjacent selected experts separated by their bounds
  float upper_rest = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (!((taken >> i) & 1u) && lane + 32 * i < E) upper_rest = fmaxf(upper_rest, v[i] + b[i]);
  upper_rest = warp_max(upper_rest);
  const float lo_sel = (lane < k) ? sel_v - sel_b : INFINITY;
  const float hi_next = __shfl_down_sync(0xffffffffu, (lane < k) ? sel_v + sel_b : -INFINITY, 1);
  const bool ordered = (lane + 1 >= k) || (lo_sel > hi_next);
  const float min_lo = -warp_max(-lo_sel);
  const bool certified = __all_sync(0xffffffffu, ordered) && (k == E || min_lo > upper_rest) &&
                         isfinite(min_lo);
  if (!certified) return false;
  const float l0 = __shfl_sync(0xffffffffu, sel_v, 0);
  const float ex = (lane < k) ? __expf(sel_v - l0) : 0.f;
  const float z = warp_sum(ex);
  if (lane < k) {
    a.idx[t * k + lane] = sel_e;
    a.wts[t * k + lane] = ex / z;
    idx_s[t * k + lane] = sel_e;
  }
  return true;
}

template <int EPL, int NW>
__global__ void __launch_bounds__(32 * NW, 1) route_select_small_kernel(RouteSmallArgs r) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const SelectArgs &a = r.sel;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int64_t E = a.E, T = a.T, nch = a.H / 128;
  const int k = a.k;
  // shared memory: [NW] exact-path scratch (E doubles + 2E floats), the sort's
  // scratch, the selected experts [T k]
  double *lg64 = reinterpret_cast<double *>(smem_raw) + (size_t)wid * E;
  float *lg = reinterpret_cast<float *>(smem_raw + (size_t)NW * E * sizeof(double)) + (size_t)wid * 2 * E;
  int *sort_smem = reinterpret_cast<int *>(smem_raw + (size_t)NW * E * (sizeof(double) + 2 * sizeof(float)));
  int32_t *idx_s = sort_smem + cta_sort_smem(NW, (int)E) / sizeof(int);
  pdl_wait();  // logits, norms and activation units come from the previous kernel
  pdl_trigger();
  for (int64_t t = wid; t < T; t += NW) {
    float ss = 0.f;
    for (int64_t c = lane; c < nch; c += 32) ss += __ldcg(r.xss + t * nch + c);
    const float xn = sqrtf(warp_sum(ss));
    if (!select_fast<EPL>(a, t, xn, idx_s)) {
      select_token(a, t, xn, lg, lg + E, lg64);
      __syncwarp();
      if (lane < k) idx_s[t * k + lane] = a.idx[t * k + lane];
    }
  }
  __syncthreads();
  if (wid == 0) {
    warp_counting_sort(idx_s, (int)(T * k), (int)E, r.tile_m, r.so, sort_smem, a.err);
  } else {
    for (int i = threadIdx.x - 32; i < r.n_counters; i += blockDim.x - 32) r.counters[i] = 0;
  }
}

// f16 copies of every token (the GEMV path above the fused-routing size).
__global__ void __launch_bounds__(128) x_to_f16_kernel(const __nv_bfloat16 *__restrict__ x, int64_t T,
                                                       int64_t H, __half *__restrict__ x16,
                                                       float *__restrict__ xscale) {
  const int64_t t = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  if (t >= T) return;
  float xn, amax;
  x_stats(x + t * H, H, &xn, &amax);
  x_to_f16(x + t * H, H, amax, x16 + t * H, xscale + t);
}

// ------------------------------------------------------------------ selection, T large
// One warp per token.  Shared memory per warp: E floats and E doubles.
// Warps take tokens from a global counter (zero at launch): a token whose
// selection needs the exact path costs many times a certified one, and
// those tokens fall unevenly, so a fixed token-to-warp map would leave the
// run as long as its most loaded SM.
__global__ void __launch_bounds__(128) router_select_kernel(SelectArgs a, int32_t *queue) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int wid = threadIdx.x >> 5, nw = blockDim.x >> 5, lane = threadIdx.x & 31;
  double *lg64 = reinterpret_cast<double *>(smem_raw) + (size_t)wid * a.E;
  float *lg = reinterpret_cast<float *>(smem_raw + (size_t)nw * a.E * sizeof(double)) + (size_t)wid * 2 * a.E;
  while (true) {
    int64_t t = 0;
    if (lane == 0) t = atomicAdd(queue, 1);
    t = __shfl_sync(0xffffffffu, t, 0);
    if (t >= a.T) break;
    float xn, amax;
    x_stats(a.x + t * a.H, a.H, &xn, &amax);
    select_token(a, t, xn, lg, lg + a.E, lg64);
  }
}

// ------------------------------------------------------------------ logits, T large
// (the tensor-core kernel in router_tc.cu; the row norms of its bound here)
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

// ------------------------------------------------------------------ launchers

// Longest rounding chain of a logit of the warp-per-expert kernel (T <=
// kRouterWarpMaxT): lane chain 4 ceil(H / 1024), butterfly 5, sum over the 8
// warps, bias.  (Large batches use the tensor-core kernel and its own bound.)
int router_chain_depth(int64_t H) { return (int)(4 * ((H + 1023) / 1024) + 5 + 8 + 1); }

float router_gamma(int64_t H) {
  const double u = 1.0 / 16777216.0;  // 2^-24
  const double d = (double)router_chain_depth(H);
  const double g = d * u / (1.0 - d * u);
  return nextafterf((float)(g * (1.0 + 1e-6)), INFINITY);
}

static SelectArgs select_args(const __nv_bfloat16 *x, int64_t T, const float *W, const float *bias,
                              int64_t E, int64_t H, int k, const float *logits, int ks,
                              const float *wnorm, float gamma, int32_t *idx, float *wts, int *err) {
  SelectArgs a;
  a.x = x; a.T = T; a.W = W; a.bias = bias; a.E = E; a.H = H; a.k = k;
  a.logits = logits; a.ks = ks; a.wnorm = wnorm; a.gamma = gamma;
  a.idx = idx; a.wts = wts; a.err = err;
  return a;
}

size_t route_decode_smem(int64_t E) {
  const size_t sel = (size_t)kRouteWarps * E * (sizeof(double) + 2 * sizeof(float));
  const size_t srt = cta_sort_smem(kRouteWarps, (int)E);
  return sel > srt ? sel : srt;
}

cudaError_t launch_route_decode(const __nv_bfloat16 *x, int64_t T, const float *W, const float *bias,
                                int64_t E, int64_t H, int k, float gamma, float *logits, float *wnorm,
                                float *xnorm, __half *x16, float *xscale, int32_t *ticket,
                                int32_t *idx, float *wts, int32_t *counts, int32_t *offsets,
                                int32_t *perm, int32_t *inv, int32_t *active, int32_t *n_active,
                                int32_t *tile_offsets, int tile_m, uint32_t *pos_max, int *err,
                                cudaStream_t s) {
  SelectArgs a = select_args(x, T, W, bias, E, H, k, logits, 1, wnorm, gamma, idx, wts, err);
  SortOut so{counts, offsets, perm, inv, active, n_active, tile_offsets};
  const size_t smem = route_decode_smem(E);
  cudaError_t e;
  if (T <= 1) {
    auto kern = route_decode_kernel<1>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess) return e;
    kern<<<(unsigned)E, 32 * kRouteWarps, smem, s>>>(a, logits, wnorm, xnorm, x16, xscale, ticket, tile_m, so, pos_max);
  } else {
    auto kern = route_decode_kernel<8>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess) return e;
    kern<<<(unsigned)E, 32 * kRouteWarps, smem, s>>>(a, logits, wnorm, xnorm, x16, xscale, ticket, tile_m, so, pos_max);
  }
  return cudaGetLastError();
}

int route_small_epc(int64_t E) { return E <= 128 ? 1 : (E <= 256 ? 2 : (E <= 512 ? 4 : 8)); }

float route_small_gamma(int64_t H, int64_t E) {
  const int wpe = kRouteWarps / route_small_epc(E);
  int lg = 0;
  while ((1 << lg) < wpe) ++lg;
  const int64_t nch_w = (H / 128 + wpe - 1) / wpe;
  const double u = 1.0 / 16777216.0;  // 2^-24
  const double d = (double)(nch_w + 2 + 5 + lg + 1);
  const double g = d * u / (1.0 - d * u);
  return nextafterf((float)(g * (1.0 + 1e-6)), INFINITY);
}

namespace {
template <int EPL, int NW>
cudaError_t launch_select_small(const RouteSmallArgs &r, cudaStream_t s) {
  const int64_t E = r.sel.E;
  const size_t smem = (size_t)NW * E * (sizeof(double) + 2 * sizeof(float)) + cta_sort_smem(NW, (int)E) +
                      (size_t)r.sel.T * r.sel.k * sizeof(int32_t);
  auto kern = route_select_small_kernel<EPL, NW>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(1), dim3(32 * NW), smem, s, r);
}
}  // namespace

cudaError_t launch_route_small(const __nv_bfloat16 *x, int64_t T, const float *W, const float *bias,
                               int64_t E, int64_t H, int k, float *logits, float *wnorm, float *xss,
                               uint8_t *a_hi, uint8_t *a_lo, float *a_scale, int64_t a_ld,
                               int32_t *counters, int n_counters, int32_t *idx,
                               float *wts, int32_t *counts, int32_t *offsets, int32_t *perm,
                               int32_t *inv, int32_t *active, int32_t *n_active,
                               int32_t *tile_offsets, int tile_m, int *err, cudaStream_t s) {
  RouteSmallArgs r;
  r.sel = select_args(x, T, W, bias, E, H, k, logits, 1, wnorm, route_small_gamma(H, E), idx, wts, err);
  r.epc = route_small_epc(E);
  r.logits_w = logits;
  r.wnorm_w = wnorm;
  r.xss = xss;
  r.a_hi = a_hi;
  r.a_lo = a_lo;
  r.a_scale = a_scale;
  r.a_ld = a_ld;
  r.counters = counters;
  r.n_counters = n_counters;
  r.tile_m = tile_m;
  r.so = SortOut{counts, offsets, perm, inv, active, n_active, tile_offsets};
  dim3 grid((unsigned)((E + r.epc - 1) / r.epc), (unsigned)((T + kSmallTB - 1) / kSmallTB));
  route_logits_small_kernel<<<grid, 32 * kRouteWarps, 0, s>>>(r);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (E <= 32) return launch_select_small<1, 16>(r, s);
  if (E <= 64) return launch_select_small<2, 16>(r, s);
  if (E <= 128) return launch_select_small<4, 16>(r, s);
  if (E <= 256) return launch_select_small<8, 16>(r, s);
  if (E <= 512) return launch_select_small<16, 16>(r, s);
  return launch_select_small<32, 8>(r, s);
}

cudaError_t launch_row_norms(const float *W, int64_t E, int64_t H, float *wnorm, cudaStream_t s) {
  row_norm_kernel<<<(unsigned)((E + 3) / 4), 128, 0, s>>>(W, E, H, wnorm);
  return cudaGetLastError();
}


cudaError_t launch_x_to_f16(const __nv_bfloat16 *x, int64_t T, int64_t H, __half *x16, float *xscale,
                           cudaStream_t s) {
  x_to_f16_kernel<<<(unsigned)((T + 3) / 4), 128, 0, s>>>(x, T, H, x16, xscale);
  return cudaGetLastError();
}

size_t router_select_smem(int64_t E) { return (size_t)4 * E * (sizeof(double) + 2 * sizeof(float)); }

cudaError_t launch_router_select(const __nv_bfloat16 *x, int64_t T, const float *W,
                                 const float *bias, int64_t E, int64_t H, int k,
                                 const float *logits, const float *wnorm, int ks, float gamma_d,
                                 int32_t *idx, float *wts, int32_t *queue, int *err, int sms,
                                 cudaStream_t s) {
  SelectArgs a = select_args(x, T, W, bias, E, H, k, logits, ks, wnorm, gamma_d, idx, wts, err);
  const size_t smem = router_select_smem(E);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(router_select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, router_select_kernel, 128, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  int64_t grid = (T + 3) / 4;
  if (grid > (int64_t)sms * per_sm) grid = (int64_t)sms * per_sm;
  if (grid <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(queue, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  router_select_kernel<<<(unsigned)grid, 128, smem, s>>>(a, queue);
  return cudaGetLastError();
}

}  // namespace fp8moe
