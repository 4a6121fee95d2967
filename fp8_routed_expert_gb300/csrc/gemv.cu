// Grouped GEMV of the routed experts for small batches (decode).
//
// Memory-bound: every active expert's e4m3 bytes are read once (the pages'
// finding that the bytes moved per token decide MoE speed: dragon.c §8
// "Round 1", DeepSeek-V4.1-Flash post "Bytes per token decide everything").
// The kernels read e4m3 codes with coalesced 16-byte loads and convert them to
// f16 in registers (never materialising dequantised weights: dragon.c §8
// "Round 2"; WARP BACKENDS.md "Never dequantize an expert"); the exact f16
// codes feed mma.sync.m16n8k16 with f32 accumulation, whose N=8 columns are up
// to 8 tokens of one expert, so one weight row serves every token routed to
// that expert (Trochilus, "Acknowledgements": one weight row against several
// tokens).  Each 128-wide K block is accumulated separately and multiplied by
// its block scale once (dragon.c §8 "Round 3": the 128-column scale is folded
// out of the inner loop).
//
// Fragment mapping.  Lane (g = lane/4, q = lane%4) loads 16 consecutive codes
// of weight rows g and g+8 at K offset 64c + 16q of a 128-wide block.  Inside a
// 64-wide chunk, k-step s (0..3) uses codes 4s..4s+3 of those 16: codes
// (4s, 4s+1) are the MMA's logical k = (2q, 2q+1) and codes (4s+2, 4s+3) are
// k = (2q+8, 2q+9).  The B operand (activations) is loaded with the same
// mapping, so the dot products are unchanged; only the order of terms inside
// each 64-wide chunk differs from the natural one.
#include "common.cuh"
#include "kernels.h"

namespace fp8moe {

// ---------------------------------------------------------------- W13 + SwiGLU
// Item = (active expert, 32 consecutive h outputs).  Warp w handles h rows
// i0 = 8 (w % 4) .. +7 of the item: MMA rows 0..7 are gate rows i0.., rows
// 8..15 the matching up rows I + i0.., so each lane ends with gate and up of
// the same (h row, token) and applies SwiGLU itself.  Warps 0-3 take the first
// half of the K blocks, warps 4-7 the second; the halves are added in shared
// memory in a fixed order.
template <int NT>
__global__ void __launch_bounds__(256) gemv13_swiglu_kernel(
    const uint8_t *__restrict__ w13, const float *__restrict__ s13, const __half *__restrict__ x16,
    const float *__restrict__ xscale, const int32_t *__restrict__ counts,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm,
    const int32_t *__restrict__ active, const int32_t *__restrict__ n_active, int k, int64_t H,
    int64_t I, float *__restrict__ h, uint32_t *__restrict__ hmax) {
  __shared__ float red[4][32][NT][4];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int tile = wid & 3, half = wid >> 2;
  const int64_t nkb = H / 128;
  const int64_t kb_mid = (nkb + 1) / 2;
  const int64_t kb_begin = half ? kb_mid : 0, kb_end = half ? nkb : kb_mid;
  const int64_t items_per_expert = I / 32;
  const int64_t n_items = (int64_t)(*n_active) * items_per_expert;
  const int64_t srow = 2 * I / 128;

  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int e = active[item / items_per_expert];
    const int64_t i0 = (item % items_per_expert) * 32 + tile * 8;
    const int64_t cnt = counts[e], seg = offsets[e];
    const uint8_t *wg_row = w13 + ((int64_t)e * 2 * I + i0 + g) * H + q * 16;
    const uint8_t *wu_row = w13 + ((int64_t)e * 2 * I + I + i0 + g) * H + q * 16;
    const float *sg = s13 + ((int64_t)e * srow + i0 / 128) * nkb;
    const float *su = s13 + ((int64_t)e * srow + (I + i0) / 128) * nkb;

    for (int64_t tb = 0; tb < cnt; tb += NT * 8) {
      const __half *xrow[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int64_t ti = tb + j * 8 + g;
        xrow[j] = (ti < cnt) ? x16 + (int64_t)(perm[seg + ti] / k) * H + q * 16 : nullptr;
      }
      float tot[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int v = 0; v < 4; ++v) tot[j][v] = 0.f;

      uint4 cg0, cg1, cu0, cu1;
      if (kb_begin < kb_end) {
        cg0 = ld_stream16(wg_row + kb_begin * 128);
        cg1 = ld_stream16(wg_row + kb_begin * 128 + 64);
        cu0 = ld_stream16(wu_row + kb_begin * 128);
        cu1 = ld_stream16(wu_row + kb_begin * 128 + 64);
      }
      for (int64_t kb = kb_begin; kb < kb_end; ++kb) {
        uint4 ng0, ng1, nu0, nu1;
        if (kb + 1 < kb_end) {
          ng0 = ld_stream16(wg_row + (kb + 1) * 128);
          ng1 = ld_stream16(wg_row + (kb + 1) * 128 + 64);
          nu0 = ld_stream16(wu_row + (kb + 1) * 128);
          nu1 = ld_stream16(wu_row + (kb + 1) * 128 + 64);
        }
        float acc[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int v = 0; v < 4; ++v) acc[j][v] = 0.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint4 wg = c ? cg1 : cg0, wu = c ? cu1 : cu0;
          uint4 xf[NT][2];
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            if (xrow[j] != nullptr) {
              xf[j][0] = ld_ro16(xrow[j] + kb * 128 + c * 64);
              xf[j][1] = ld_ro16(xrow[j] + kb * 128 + c * 64 + 8);
            } else {
              xf[j][0] = make_uint4(0, 0, 0, 0);
              xf[j][1] = make_uint4(0, 0, 0, 0);
            }
          }
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint32_t gw = u4_word(wg, s), uw = u4_word(wu, s);
            const uint32_t a0 = e4m3x2_to_f16x2(gw & 0xffffu);
            const uint32_t a1 = e4m3x2_to_f16x2(uw & 0xffffu);
            const uint32_t a2 = e4m3x2_to_f16x2(gw >> 16);
            const uint32_t a3 = e4m3x2_to_f16x2(uw >> 16);
#pragma unroll
            for (int j = 0; j < NT; ++j)
              mma_16816(acc[j], a0, a1, a2, a3, u4_word(xf[j][s >> 1], (2 * s) & 3),
                        u4_word(xf[j][s >> 1], (2 * s + 1) & 3));
          }
        }
        const float scg = __ldg(sg + kb), scu = __ldg(su + kb);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          tot[j][0] = fmaf(acc[j][0], scg, tot[j][0]);
          tot[j][1] = fmaf(acc[j][1], scg, tot[j][1]);
          tot[j][2] = fmaf(acc[j][2], scu, tot[j][2]);
          tot[j][3] = fmaf(acc[j][3], scu, tot[j][3]);
        }
        cg0 = ng0; cg1 = ng1; cu0 = nu0; cu1 = nu1;
      }

      if (half == 1) {
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int v = 0; v < 4; ++v) red[tile][lane][j][v] = tot[j][v];
      }
      __syncthreads();
      if (half == 0) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
#pragma unroll
          for (int d = 0; d < 2; ++d) {
            const int64_t ti = tb + j * 8 + 2 * q + d;
            if (ti >= cnt) continue;
            const int64_t pos = seg + ti;
            const float xs = xscale[perm[pos] / k];
            const float gv = (tot[j][d] + red[tile][lane][j][d]) * xs;
            const float uv = (tot[j][2 + d] + red[tile][lane][j][2 + d]) * xs;
            const float hv = swiglu(gv, uv);
            h[pos * I + i0 + g] = hv;
            atomicMax(&hmax[pos], __float_as_uint(fabsf(hv)));
          }
        }
      }
      __syncthreads();
    }
  }
}

// ---------------------------------------------------------------- W2
// Item = (active expert, 64 consecutive output rows).  Warp w computes rows
// j0 = 16 (w % 4) .. +15 over one half of the K blocks of I.  The activations
// h (f32) are split into an f16 pair hi + lo after an exact power-of-two
// scaling chosen from the position's largest |h|, so the products keep about
// 22 bits of h.
template <int NT>
__global__ void __launch_bounds__(256) gemv2_kernel(
    const uint8_t *__restrict__ w2, const float *__restrict__ s2, const float *__restrict__ h,
    const uint32_t *__restrict__ hmax, const int32_t *__restrict__ counts,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ active,
    const int32_t *__restrict__ n_active, int64_t H, int64_t I, float *__restrict__ y) {
  __shared__ float red[4][32][NT][4];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  const int tile = wid & 3, half = wid >> 2;
  const int64_t nkb = I / 128;
  const int64_t kb_mid = (nkb + 1) / 2;
  const int64_t kb_begin = half ? kb_mid : 0, kb_end = half ? nkb : kb_mid;
  const int64_t items_per_expert = H / 64;
  const int64_t n_items = (int64_t)(*n_active) * items_per_expert;

  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int e = active[item / items_per_expert];
    const int64_t j0 = (item % items_per_expert) * 64 + tile * 16;
    const int64_t cnt = counts[e], seg = offsets[e];
    const uint8_t *wa_row = w2 + ((int64_t)e * H + j0 + g) * I + q * 16;
    const uint8_t *wb_row = w2 + ((int64_t)e * H + j0 + 8 + g) * I + q * 16;
    const float *sc = s2 + ((int64_t)e * (H / 128) + j0 / 128) * nkb;

    for (int64_t tb = 0; tb < cnt; tb += NT * 8) {
      const float *hrow[NT];
      float down[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int64_t ti = tb + j * 8 + g;
        hrow[j] = (ti < cnt) ? h + (seg + ti) * I + q * 16 : nullptr;
        down[j] = (ti < cnt) ? exp2i(-f16_range_shift(__uint_as_float(hmax[seg + ti]))) : 0.f;
      }
      float tot[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int v = 0; v < 4; ++v) tot[j][v] = 0.f;

      uint4 ca0, ca1, cb0, cb1;
      if (kb_begin < kb_end) {
        ca0 = ld_stream16(wa_row + kb_begin * 128);
        ca1 = ld_stream16(wa_row + kb_begin * 128 + 64);
        cb0 = ld_stream16(wb_row + kb_begin * 128);
        cb1 = ld_stream16(wb_row + kb_begin * 128 + 64);
      }
      for (int64_t kb = kb_begin; kb < kb_end; ++kb) {
        uint4 na0, na1, nb0, nb1;
        if (kb + 1 < kb_end) {
          na0 = ld_stream16(wa_row + (kb + 1) * 128);
          na1 = ld_stream16(wa_row + (kb + 1) * 128 + 64);
          nb0 = ld_stream16(wb_row + (kb + 1) * 128);
          nb1 = ld_stream16(wb_row + (kb + 1) * 128 + 64);
        }
        float acc[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int v = 0; v < 4; ++v) acc[j][v] = 0.f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint4 wa = c ? ca1 : ca0, wb = c ? cb1 : cb0;
          uint32_t bhi[NT][8], blo[NT][8];
#pragma unroll
          for (int j = 0; j < NT; ++j) {
            if (hrow[j] != nullptr) {
              const float4 *src = reinterpret_cast<const float4 *>(hrow[j] + kb * 128 + c * 64);
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                float4 v = __ldg(src + m);
                v.x *= down[j]; v.y *= down[j]; v.z *= down[j]; v.w *= down[j];
                const uint32_t h0 = pack_f16x2(v.x, v.y), h1 = pack_f16x2(v.z, v.w);
                const float2 r0 = unpack_f16x2(h0), r1 = unpack_f16x2(h1);
                bhi[j][2 * m] = h0;
                bhi[j][2 * m + 1] = h1;
                blo[j][2 * m] = pack_f16x2(v.x - r0.x, v.y - r0.y);
                blo[j][2 * m + 1] = pack_f16x2(v.z - r1.x, v.w - r1.y);
              }
            } else {
#pragma unroll
              for (int m = 0; m < 8; ++m) { bhi[j][m] = 0u; blo[j][m] = 0u; }
            }
          }
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint32_t aw = u4_word(wa, s), bw = u4_word(wb, s);
            const uint32_t a0 = e4m3x2_to_f16x2(aw & 0xffffu);
            const uint32_t a1 = e4m3x2_to_f16x2(bw & 0xffffu);
            const uint32_t a2 = e4m3x2_to_f16x2(aw >> 16);
            const uint32_t a3 = e4m3x2_to_f16x2(bw >> 16);
#pragma unroll
            for (int j = 0; j < NT; ++j) {
              mma_16816(acc[j], a0, a1, a2, a3, bhi[j][2 * s], bhi[j][2 * s + 1]);
              mma_16816(acc[j], a0, a1, a2, a3, blo[j][2 * s], blo[j][2 * s + 1]);
            }
          }
        }
        const float sck = __ldg(sc + kb);
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int v = 0; v < 4; ++v) tot[j][v] = fmaf(acc[j][v], sck, tot[j][v]);
        ca0 = na0; ca1 = na1; cb0 = nb0; cb1 = nb1;
      }

      if (half == 1) {
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int v = 0; v < 4; ++v) red[tile][lane][j][v] = tot[j][v];
      }
      __syncthreads();
      if (half == 0) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
#pragma unroll
          for (int d = 0; d < 2; ++d) {
            const int64_t ti = tb + j * 8 + 2 * q + d;
            if (ti >= cnt) continue;
            const int64_t pos = seg + ti;
            const float up = exp2i(f16_range_shift(__uint_as_float(hmax[pos])));
            y[pos * H + j0 + g] = (tot[j][d] + red[tile][lane][j][d]) * up;
            y[pos * H + j0 + 8 + g] = (tot[j][2 + d] + red[tile][lane][j][2 + d]) * up;
          }
        }
      }
      __syncthreads();
    }
  }
}

// ---------------------------------------------------------------- combine
// out[t, :] = bf16_rne( sum_{r=0}^{k-1} w[t, r] * y[inv[t k + r], :] ), summed
// in router rank order with one fma chain per element (WARP BACKENDS.md,
// "Coherent memory": partials reduced in original router order) and no atomics.
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ y,
                                                      const int32_t *__restrict__ inv,
                                                      const float *__restrict__ wts, int64_t T,
                                                      int k, int64_t H,
                                                      __nv_bfloat16 *__restrict__ out) {
  const int64_t t = blockIdx.x;
  if (t >= T) return;
  for (int64_t j = 4 * (int64_t)(blockIdx.y * blockDim.x + threadIdx.x); j < H;
       j += 4 * (int64_t)blockDim.x * gridDim.y) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = 0; r < k; ++r) {
      const int64_t pos = inv[t * k + r];
      const float w = wts[t * k + r];
      const float4 v = __ldg(reinterpret_cast<const float4 *>(y + pos * H + j));
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t *>(&lo);
    o.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(out + t * H + j) = o;
  }
}

// ---------------------------------------------------------------- launchers

cudaError_t launch_gemv13(const uint8_t *w13, const float *s13, const __half *x16,
                          const float *xscale, const int32_t *counts, const int32_t *offsets,
                          const int32_t *perm, const int32_t *active, const int32_t *n_active,
                          int k, int64_t H, int64_t I, float *h, uint32_t *hmax, int64_t max_items,
                          int wide_tokens, int grid_cap, cudaStream_t s) {
  const int64_t grid = max_items < grid_cap ? max_items : grid_cap;
  if (grid <= 0) return cudaSuccess;
  if (wide_tokens)
    gemv13_swiglu_kernel<4><<<(unsigned)grid, 256, 0, s>>>(w13, s13, x16, xscale, counts, offsets,
                                                           perm, active, n_active, k, H, I, h, hmax);
  else
    gemv13_swiglu_kernel<1><<<(unsigned)grid, 256, 0, s>>>(w13, s13, x16, xscale, counts, offsets,
                                                           perm, active, n_active, k, H, I, h, hmax);
  return cudaGetLastError();
}

cudaError_t launch_gemv2(const uint8_t *w2, const float *s2, const float *h, const uint32_t *hmax,
                         const int32_t *counts, const int32_t *offsets, const int32_t *active,
                         const int32_t *n_active, int64_t H, int64_t I, float *y,
                         int64_t max_items, int wide_tokens, int grid_cap, cudaStream_t s) {
  const int64_t grid = max_items < grid_cap ? max_items : grid_cap;
  if (grid <= 0) return cudaSuccess;
  if (wide_tokens)
    gemv2_kernel<4><<<(unsigned)grid, 256, 0, s>>>(w2, s2, h, hmax, counts, offsets, active,
                                                   n_active, H, I, y);
  else
    gemv2_kernel<1><<<(unsigned)grid, 256, 0, s>>>(w2, s2, h, hmax, counts, offsets, active,
                                                   n_active, H, I, y);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float *y, const int32_t *inv, const float *wts, int64_t T, int k,
                           int64_t H, __nv_bfloat16 *out, cudaStream_t s) {
  dim3 grid((unsigned)T, (unsigned)((H + 1023) / 1024));
  combine_kernel<<<grid, 256, 0, s>>>(y, inv, wts, T, k, H, out);
  return cudaGetLastError();
}

}  // namespace fp8moe
