// Routed experts with FP4 (NVFP4) weights for small batches: grouped GEMVs
// that read the packed codes once and dequantise them in registers.
//
// Format (the Qwen post's experts, "Why this model" and "The engine", piece
// 1): e2m1 codes, two per byte along K with the even element in the low
// nibble; one e4m3 scale per 16 consecutive weights of a row; one f32 global
// scale per expert matrix.  A weight is e2m1 * e4m3 scale * global.
//
// Decode is bound by the bytes of the selected experts (DeepSeek-V4.1-Flash
// post, "Bytes per token decide everything"); FP4 halves them against FP8.
// Each lane converts its codes with the hardware e2m1x2 -> f16x2 conversion
// (the Qwen post's expert kernel uses the same instruction) and multiplies
// them by their group's scale in f16: an e2m1 value (2 significant bits)
// times an e4m3 scale (4 bits) is exact in f16, so the A operand of
// mma.sync.m16n8k16 carries the exact weight / global.  The global scale and
// the activations' power-of-two range shift are applied to the f32 result.
//
// Fragment mapping (one warp, 16 weight rows x 8 positions per MMA).  Lane
// (g = lane / 4, q = lane % 4) loads 16 bytes (32 codes) of rows g and g + 8
// at K offset 32 q of each 128-wide chunk: two whole 16-weight scale groups
// (2 q, 2 q + 1 of the chunk's 8).  K step s (0..7) of the chunk uses the
// lane's codes 4 s .. 4 s + 3: codes (4 s, 4 s + 1) are the MMA's logical
// k = (2 q, 2 q + 1), codes (4 s + 2, 4 s + 3) are k = (2 q + 8, 2 q + 9).
// The B operand (activations) is read with the same mapping -- 8 contiguous
// bytes of f16 per lane and step -- so the dot products are those of the
// natural K order with the terms regrouped.
#include "common.cuh"
#include "kernels.h"

namespace fp8moe {

namespace {

constexpr int kFp4Warps = 4;   // warps per CTA
constexpr int kStageRows = 8;  // positions staged in shared memory per pass (NG = 1)

// Shared memory of a CTA for NG = 1: the activation rows of the pass's 8
// positions as f16, rows padded by 16 bytes against bank conflicts (gate/up:
// x; down: h as a hi and a lo plane).
__host__ __device__ constexpr int64_t stage_pitch(int64_t K) { return K + 8; }
__host__ __device__ constexpr size_t stage_bytes(int64_t K, int planes) {
  return (size_t)planes * kStageRows * stage_pitch(K) * 2;
}

// Four bytes of packed e2m1 pairs -> four f16x2 (element 2j in the low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t codes, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\tmov.b32 {c0, c1, c2, c3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, c0;\n\tcvt.rn.f16x2.e2m1x2 %1, c1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, c2;\n\tcvt.rn.f16x2.e2m1x2 %3, c3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(codes));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
  return *reinterpret_cast<uint32_t *>(&r);
}

// The two e4m3 group scales of a lane (low byte: group 2q, high: 2q + 1) as
// two broadcast f16x2 values.
__device__ __forceinline__ void group_scales(uint32_t two, uint32_t &s0, uint32_t &s1) {
  const uint32_t h = e4m3x2_to_f16x2(two & 0xffffu);
  s0 = (h & 0xffffu) | (h << 16);
  s1 = (h >> 16) | (h & 0xffff0000u);
}

__device__ __forceinline__ uint32_t ld_u16(const uint8_t *p) {
  return (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(p));
}

// Converts one chunk's codes of rows g (wa) and g + 8 (wb) into the A
// registers of its 8 K steps: a[s][0..3].
__device__ __forceinline__ void chunk_fragments(const uint4 &wa, const uint4 &wb, uint32_t sca,
                                                uint32_t scb, uint32_t (&a)[8][4]) {
  uint32_t sa0, sa1, sb0, sb1;
  group_scales(sca, sa0, sa1);
  group_scales(scb, sb0, sb1);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t ha[4], hb[4];
    e2m1x8_to_f16x2(u4_word(wa, w), ha);  // codes 8w .. 8w + 7 of row g
    e2m1x8_to_f16x2(u4_word(wb, w), hb);
    const uint32_t ga = w < 2 ? sa0 : sa1, gb = w < 2 ? sb0 : sb1;
#pragma unroll
    for (int hs = 0; hs < 2; ++hs) {  // step s = 2 w + hs: codes 4 s .. 4 s + 3
      const int s = 2 * w + hs;
      a[s][0] = hmul2_u32(ha[2 * hs], ga);      // row g, codes 4s, 4s+1
      a[s][1] = hmul2_u32(hb[2 * hs], gb);      // row g + 8
      a[s][2] = hmul2_u32(ha[2 * hs + 1], ga);  // row g, codes 4s+2, 4s+3
      a[s][3] = hmul2_u32(hb[2 * hs + 1], gb);
    }
  }
}

// ---------------------------------------------------------------- W13 + SwiGLU
// Item = (active expert, 8 consecutive h outputs i0..i0+7), one warp, all of
// K = H: MMA rows 0..7 are gate rows i0.., rows 8..15 the up rows I + i0..,
// so a lane ends with gate and up of the same (h output, position).  NG
// groups of 8 positions share each converted weight chunk; experts with more
// positions take further passes.
// U: 128-wide K chunks whose weight loads are issued together; PIPE: two
// register sets, the next U chunks' loads in flight while these are used.
template <int NG, int U, bool PIPE>
__global__ void __launch_bounds__(32 * kFp4Warps) fp4_gate_up_kernel(
    const uint8_t *__restrict__ w13, const uint8_t *__restrict__ sf13, const float *__restrict__ g13,
    const __half *__restrict__ x16, const float *__restrict__ xscale,
    const int32_t *__restrict__ counts, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ perm, const int32_t *__restrict__ active,
    const int32_t *__restrict__ n_active, int k, int64_t H, int64_t I, float *__restrict__ h,
    uint32_t *__restrict__ hmax) {
  extern __shared__ __align__(16) __half xs[];  // NG = 1: [kStageRows][stage_pitch(H)]
  pdl_wait();  // routing, x16 and the cleared maxima come from the previous kernel
  pdl_trigger();
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int64_t ipe = I / 8, n_items = (int64_t)*n_active * ipe;
  const int64_t nkc = H / 128, pitch = stage_pitch(H);
  const int64_t n_warps = (int64_t)gridDim.x * kFp4Warps;
  // rounds of kFp4Warps consecutive items, one per warp: the CTA's items of a
  // round belong to one expert (kFp4Warps divides the items per expert), so
  // for NG = 1 the CTA stages that expert's activation rows once per pass
  for (int64_t base = (int64_t)blockIdx.x * kFp4Warps; base < n_items; base += n_warps) {
    const int64_t item = base + (threadIdx.x >> 5);
    const bool has = item < n_items;
    const int e = active[base / ipe];
    const int64_t i0 = (item % ipe) * 8;
    const int64_t rg = (int64_t)e * 2 * I + i0 + g, ru = rg + I;  // gate and up rows
    const uint8_t *wg = w13 + rg * (H / 2) + 16 * q, *wu = w13 + ru * (H / 2) + 16 * q;
    const uint8_t *sg = sf13 + rg * (H / 16) + 2 * q, *su = sf13 + ru * (H / 16) + 2 * q;
    const int cnt = counts[e], off = offsets[e];
    const float ge = g13[e];
    for (int n0 = 0; n0 < cnt; n0 += 8 * NG) {
      const int ngroups = (cnt - n0 + 7) / 8;  // groups of 8 positions with work in this pass
      // B rows: position n0 + 8 ng + g of this pass (a zero row past the segment)
      const __half *xr[NG];
      if constexpr (NG == 1) {
        __syncthreads();  // the previous pass's reads are done
        const int64_t row8 = H / 8;
        for (int64_t i = threadIdx.x; i < kStageRows * row8; i += blockDim.x) {
          const int r = (int)(i / row8);
          const int64_t c8 = i - r * row8;
          const int n = n0 + r;
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (n < cnt) v = __ldg(reinterpret_cast<const uint4 *>(x16 + (int64_t)(perm[off + n] / k) * H) + c8);
          *reinterpret_cast<uint4 *>(xs + r * pitch + 8 * c8) = v;
        }
        __syncthreads();
        xr[0] = xs + g * pitch + 32 * q;
      } else {
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          const int n = n0 + 8 * ng + g;
          xr[ng] = n < cnt ? x16 + (int64_t)(perm[off + n] / k) * H + 32 * q : nullptr;
        }
      }
      if (!has) continue;
      float acc[NG][4];
#pragma unroll
      for (int ng = 0; ng < NG; ++ng)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[ng][i] = 0.f;
      auto load = [&](int64_t kc0, uint4 (&wa)[U], uint4 (&wb)[U], uint32_t (&sca)[U], uint32_t (&scb)[U]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (kc0 + u < nkc) {
            wa[u] = ld_stream16(wg + (kc0 + u) * 64);
            wb[u] = ld_stream16(wu + (kc0 + u) * 64);
            sca[u] = ld_u16(sg + (kc0 + u) * 8);
            scb[u] = ld_u16(su + (kc0 + u) * 8);
          }
        }
      };
      auto comp = [&](int64_t kc0, const uint4 (&wa)[U], const uint4 (&wb)[U], const uint32_t (&sca)[U],
                      const uint32_t (&scb)[U]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (kc0 + u >= nkc) break;
          uint32_t a[8][4];
          chunk_fragments(wa[u], wb[u], sca[u], scb[u], a);
#pragma unroll
          for (int ng = 0; ng < NG; ++ng) {
            if (ng >= ngroups) break;  // warp-uniform: groups past the segment hold no position
            const __half *xp = xr[ng] ? xr[ng] + (kc0 + u) * 128 : nullptr;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
              uint2 b;
              if constexpr (NG == 1) b = *reinterpret_cast<const uint2 *>(xp + 4 * s);
              else b = xp ? __ldg(reinterpret_cast<const uint2 *>(xp + 4 * s)) : make_uint2(0u, 0u);
              mma_16816(acc[ng], a[s][0], a[s][1], a[s][2], a[s][3], b.x, b.y);
            }
          }
        }
      };
      uint4 wa0[U], wb0[U];
      uint32_t sa0[U], sb0[U];
      if constexpr (PIPE) {
        uint4 wa1[U], wb1[U];
        uint32_t sa1[U], sb1[U];
        load(0, wa0, wb0, sa0, sb0);
        for (int64_t kc0 = 0; kc0 < nkc; kc0 += 2 * U) {
          if (kc0 + U < nkc) load(kc0 + U, wa1, wb1, sa1, sb1);
          comp(kc0, wa0, wb0, sa0, sb0);
          if (kc0 + U >= nkc) break;
          if (kc0 + 2 * U < nkc) load(kc0 + 2 * U, wa0, wb0, sa0, sb0);
          comp(kc0 + U, wa1, wb1, sa1, sb1);
        }
      } else {
        for (int64_t kc0 = 0; kc0 < nkc; kc0 += U) {
          load(kc0, wa0, wb0, sa0, sb0);
          comp(kc0, wa0, wb0, sa0, sb0);
        }
      }
      // c0, c1: gate of output i0 + g for positions 8 ng + 2q, + 1; c2, c3: up
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int n = n0 + 8 * ng + 2 * q + c;
          if (n < cnt) {
            const int64_t pos = off + n;
            const float sx = ge * xscale[perm[pos] / k];
            const float hv = swiglu(acc[ng][c] * sx, acc[ng][2 + c] * sx);
            h[pos * I + i0 + g] = hv;
            atomicMax(hmax + pos, __float_as_uint(fabsf(hv)));
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------- W2
// Item = (active expert, 16 consecutive output rows j0..j0+15), one warp, all
// of K = I.  B = h of the expert's positions as an f16 hi / lo pair after an
// exact power-of-two shift per position (two MMAs into one accumulator).
// U: 128-wide K chunks whose weight loads are issued together.
template <int NG, int U>
__global__ void __launch_bounds__(32 * kFp4Warps) fp4_down_kernel(
    const uint8_t *__restrict__ w2, const uint8_t *__restrict__ sf2, const float *__restrict__ g2,
    const float *__restrict__ h, const uint32_t *__restrict__ hmax,
    const int32_t *__restrict__ counts, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ active, const int32_t *__restrict__ n_active, int64_t H, int64_t I,
    float *__restrict__ y) {
  // NG = 1: the pass's h rows, shifted, as an f16 hi plane then a lo plane
  extern __shared__ __align__(16) __half hs[];
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int64_t ipe = H / 16, n_items = (int64_t)*n_active * ipe;
  const int64_t nkc = I / 128, pitch = stage_pitch(I), plane = kStageRows * pitch;
  const int64_t n_warps = (int64_t)gridDim.x * kFp4Warps;
  // rounds of kFp4Warps consecutive items of one expert, as in the gate/up kernel
  for (int64_t base = (int64_t)blockIdx.x * kFp4Warps; base < n_items; base += n_warps) {
    const int64_t item = base + (threadIdx.x >> 5);
    const bool has = item < n_items;
    const int e = active[base / ipe];
    const int64_t j0 = (item % ipe) * 16;
    const int64_t ra = (int64_t)e * H + j0 + g, rb = ra + 8;
    const uint8_t *wa_p = w2 + ra * (I / 2) + 16 * q, *wb_p = w2 + rb * (I / 2) + 16 * q;
    const uint8_t *sa_p = sf2 + ra * (I / 16) + 2 * q, *sb_p = sf2 + rb * (I / 16) + 2 * q;
    const int cnt = counts[e], off = offsets[e];
    const float ge = g2[e];
    for (int n0 = 0; n0 < cnt; n0 += 8 * NG) {
      const int ngroups = (cnt - n0 + 7) / 8;
      const float *hr[NG];
      float down[NG];
      if constexpr (NG == 1) {
        __syncthreads();  // the previous pass's reads are done
        const int64_t row4 = I / 4;
        for (int64_t i = threadIdx.x; i < kStageRows * row4; i += blockDim.x) {
          const int r = (int)(i / row4);
          const int64_t c4 = i - r * row4;
          const int n = n0 + r;
          uint2 hi = make_uint2(0u, 0u), lo = make_uint2(0u, 0u);
          if (n < cnt) {
            const float d = exp2i(-f16_range_shift(__uint_as_float(hmax[off + n])));
            const float4 v = __ldg(reinterpret_cast<const float4 *>(h + (int64_t)(off + n) * I) + c4);
            const float v0 = v.x * d, v1 = v.y * d, v2 = v.z * d, v3 = v.w * d;
            hi = make_uint2(pack_f16x2(v0, v1), pack_f16x2(v2, v3));
            const float2 r0 = unpack_f16x2(hi.x), r1 = unpack_f16x2(hi.y);
            lo = make_uint2(pack_f16x2(v0 - r0.x, v1 - r0.y), pack_f16x2(v2 - r1.x, v3 - r1.y));
          }
          *reinterpret_cast<uint2 *>(hs + r * pitch + 4 * c4) = hi;
          *reinterpret_cast<uint2 *>(hs + plane + r * pitch + 4 * c4) = lo;
        }
        __syncthreads();
        hr[0] = nullptr;
        down[0] = 0.f;
      } else {
#pragma unroll
        for (int ng = 0; ng < NG; ++ng) {
          const int n = n0 + 8 * ng + g;
          hr[ng] = n < cnt ? h + (int64_t)(off + n) * I + 32 * q : nullptr;
          down[ng] = n < cnt ? exp2i(-f16_range_shift(__uint_as_float(hmax[off + n]))) : 0.f;
        }
      }
      if (!has) continue;
      float acc[NG][4];
#pragma unroll
      for (int ng = 0; ng < NG; ++ng)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[ng][i] = 0.f;
      for (int64_t kc0 = 0; kc0 < nkc; kc0 += U) {
        uint4 wa[U], wb[U];
        uint32_t sca[U], scb[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (kc0 + u < nkc) {
            wa[u] = ld_stream16(wa_p + (kc0 + u) * 64);
            wb[u] = ld_stream16(wb_p + (kc0 + u) * 64);
            sca[u] = ld_u16(sa_p + (kc0 + u) * 8);
            scb[u] = ld_u16(sb_p + (kc0 + u) * 8);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          if (kc0 + u >= nkc) break;
          uint32_t a[8][4];
          chunk_fragments(wa[u], wb[u], sca[u], scb[u], a);
          if constexpr (NG == 1) {
            const __half *hp = hs + g * pitch + (kc0 + u) * 128 + 32 * q;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
              const uint2 hi = *reinterpret_cast<const uint2 *>(hp + 4 * s);
              const uint2 lo = *reinterpret_cast<const uint2 *>(hp + plane + 4 * s);
              mma_16816(acc[0], a[s][0], a[s][1], a[s][2], a[s][3], hi.x, hi.y);
              mma_16816(acc[0], a[s][0], a[s][1], a[s][2], a[s][3], lo.x, lo.y);
            }
          } else {
#pragma unroll
            for (int ng = 0; ng < NG; ++ng) {
              if (ng >= ngroups) break;  // warp-uniform
              const float *hp = hr[ng] ? hr[ng] + (kc0 + u) * 128 : nullptr;
#pragma unroll
              for (int s = 0; s < 8; ++s) {
                const float4 v = hp ? __ldg(reinterpret_cast<const float4 *>(hp + 4 * s))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
                const float d = down[ng];
                const float v0 = v.x * d, v1 = v.y * d, v2 = v.z * d, v3 = v.w * d;
                const uint32_t hi0 = pack_f16x2(v0, v1), hi1 = pack_f16x2(v2, v3);
                const float2 r0 = unpack_f16x2(hi0), r1 = unpack_f16x2(hi1);
                const uint32_t lo0 = pack_f16x2(v0 - r0.x, v1 - r0.y), lo1 = pack_f16x2(v2 - r1.x, v3 - r1.y);
                mma_16816(acc[ng], a[s][0], a[s][1], a[s][2], a[s][3], hi0, hi1);
                mma_16816(acc[ng], a[s][0], a[s][1], a[s][2], a[s][3], lo0, lo1);
              }
            }
          }
        }
      }
      // c0, c1: row j0 + g for positions 8 ng + 2q, + 1; c2, c3: row j0 + g + 8
#pragma unroll
      for (int ng = 0; ng < NG; ++ng) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int n = n0 + 8 * ng + 2 * q + c;
          if (n < cnt) {
            const int64_t pos = off + n;
            const float up = ge * exp2i(f16_range_shift(__uint_as_float(hmax[pos])));
            y[pos * H + j0 + g] = acc[ng][c] * up;
            y[pos * H + j0 + g + 8] = acc[ng][2 + c] * up;
          }
        }
      }
    }
  }
}

template <typename K>
int64_t fp4_grid(K kernel, int64_t max_items, int sms, size_t smem) {
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 32 * kFp4Warps, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  int64_t grid = (max_items + kFp4Warps - 1) / kFp4Warps;
  const int64_t cap = (int64_t)sms * per_sm;
  return grid < cap ? grid : cap;
}

}  // namespace

cudaError_t launch_fp4_gate_up(const uint8_t *w13, const uint8_t *sf13, const float *g13,
                               const __half *x16, const float *xscale, const int32_t *counts,
                               const int32_t *offsets, const int32_t *perm, const int32_t *active,
                               const int32_t *n_active, int k, int64_t T, int64_t H, int64_t I,
                               float *h, uint32_t *hmax, int64_t max_items, int sms, cudaStream_t s) {
  if (max_items <= 0) return cudaSuccess;
  if (I % (8 * kFp4Warps) != 0) return cudaErrorInvalidValue;  // whole rounds per expert
  if (T <= 8) {
    auto kern = fp4_gate_up_kernel<1, 8, false>;
    const size_t smem = stage_bytes(H, 1);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3((unsigned)fp4_grid(kern, max_items, sms, smem)), dim3(32 * kFp4Warps), smem,
                      s, w13, sf13, g13, x16, xscale, counts, offsets, perm, active, n_active, k, H, I, h,
                      hmax);
  }
  auto kern = fp4_gate_up_kernel<4, 2, true>;
  return launch_pdl(kern, dim3((unsigned)fp4_grid(kern, max_items, sms, 0)), dim3(32 * kFp4Warps), 0, s,
                    w13, sf13, g13, x16, xscale, counts, offsets, perm, active, n_active, k, H, I, h,
                    hmax);
}

cudaError_t launch_fp4_down(const uint8_t *w2, const uint8_t *sf2, const float *g2, const float *h,
                            const uint32_t *hmax, const int32_t *counts, const int32_t *offsets,
                            const int32_t *active, const int32_t *n_active, int64_t T, int64_t H,
                            int64_t I, float *y, int64_t max_items, int sms, cudaStream_t s) {
  if (max_items <= 0) return cudaSuccess;
  if (H % (16 * kFp4Warps) != 0) return cudaErrorInvalidValue;  // whole rounds per expert
  if (T <= 8) {
    auto kern = fp4_down_kernel<1, 4>;
    const size_t smem = stage_bytes(I, 2);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3((unsigned)fp4_grid(kern, max_items, sms, smem)), dim3(32 * kFp4Warps), smem,
                      s, w2, sf2, g2, h, hmax, counts, offsets, active, n_active, H, I, y);
  }
  auto kern = fp4_down_kernel<4, 2>;
  return launch_pdl(kern, dim3((unsigned)fp4_grid(kern, max_items, sms, 0)), dim3(32 * kFp4Warps), 0, s,
                    w2, sf2, g2, h, hmax, counts, offsets, active, n_active, H, I, y);
}

}  // namespace fp8moe
