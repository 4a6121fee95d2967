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

// ---------------------------------------------------------------- staging
// Each warp owns a contiguous range of items (16 weight rows x all of K) and
// streams the rows through a private ring of shared-memory stages with 16-byte
// cp.async copies (L2 only).  A stage holds two 128-wide K blocks of the 16
// rows (4 KiB); copy instruction m moves 2 rows x 256 contiguous bytes, so
// HBM sees row-sequential 256-byte runs.  In shared memory a stage is
// [K block][row][128 bytes] with the 16-byte chunk index XORed by 4 (row & 1),
// which keeps the MMA fragment reads (8 lanes = 2 rows per phase) free of bank
// conflicts.  kRing - 1 stages (8 KiB per warp, 16 warps per SM) stay in
// flight without holding registers; the ring runs across item boundaries.

constexpr int kStageKB = 2;                          // 128-wide K blocks per stage
constexpr int kStageBytes = kStageKB * 16 * 128;    // 16 rows
constexpr int kRing = 3;
constexpr int kGemvWarps = 4;

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// byte offset of (K block kbl, row, 16-byte chunk) inside a stage
__device__ __forceinline__ int stage_off(int kbl, int row, int chunk) {
  return kbl * 2048 + row * 128 + ((chunk ^ ((row & 1) << 2)) << 4);
}

// Item range [lo, hi) of this warp: warps split the items into contiguous,
// equal (+-1) ranges.
__device__ __forceinline__ void warp_items(int n_items, int *lo, int *hi) {
  const int64_t tw = (int64_t)gridDim.x * kGemvWarps;
  const int64_t gw = (int64_t)blockIdx.x * kGemvWarps + (threadIdx.x >> 5);
  *lo = (int)((int64_t)n_items * gw / tw);
  *hi = (int)((int64_t)n_items * (gw + 1) / tw);
}

// Per-lane constants of the copy pattern: copy m (0..7) of a stage moves row
// 2m + (lane >> 4), 16-byte chunk (lane & 15) of the stage's 256 bytes.
struct CopyLane {
  int soff;  // shared-memory byte offset of copy 0 (copy m adds 256 m)
  int col;   // 16-byte chunk index 0..15 within the row's 256 bytes
  int rpar;  // row parity (lane >> 4)
};
__device__ __forceinline__ CopyLane copy_lane(int lane) {
  CopyLane c;
  c.col = lane & 15;
  c.rpar = lane >> 4;
  c.soff = stage_off(c.col >> 3, c.rpar, c.col & 7);
  return c;
}

// Converts the staged codes of one K block of rows g and g + 8 (fragment
// offsets f0, f1 for the two 64-byte halves) to the f16 A registers of the
// 8 k-steps: a[c][s][r].
__device__ __forceinline__ void stage_fragments(const uint8_t *sk, int f0, int f1,
                                                uint32_t (&a)[2][4][4]) {
  const uint4 r0 = *reinterpret_cast<const uint4 *>(sk + f0);
  const uint4 r1 = *reinterpret_cast<const uint4 *>(sk + f1);
  const uint4 s0 = *reinterpret_cast<const uint4 *>(sk + f0 + 1024);
  const uint4 s1 = *reinterpret_cast<const uint4 *>(sk + f1 + 1024);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint4 lo = c ? r1 : r0, hi = c ? s1 : s0;
#pragma unroll
    for (int s4 = 0; s4 < 4; ++s4) {
      const uint32_t lw = u4_word(lo, s4), hw = u4_word(hi, s4);
      a[c][s4][0] = e4m3x2_to_f16x2(lw & 0xffffu);
      a[c][s4][1] = e4m3x2_to_f16x2(hw & 0xffffu);
      a[c][s4][2] = e4m3x2_to_f16x2(lw >> 16);
      a[c][s4][3] = e4m3x2_to_f16x2(hw >> 16);
    }
  }
}

// ---------------------------------------------------------------- W13 + SwiGLU
// Item = (active expert, 8 consecutive h outputs i0..i0+7), one warp, all of
// K.  MMA rows 0..7 are the gate rows i0.., rows 8..15 the matching up rows
// I + i0.., so each lane ends with gate and up of the same (h row, token) and
// applies SwiGLU itself.  Columns are up to 8 tokens of the expert per MMA;
// NT groups of 8 share each staged weight chunk.
template <int NT>
__global__ void __launch_bounds__(32 * kGemvWarps) gemv13_swiglu_kernel(
    const uint8_t *__restrict__ w13, const float *__restrict__ s13, const __half *__restrict__ x16,
    const float *__restrict__ xscale, const int32_t *__restrict__ counts,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm,
    const int32_t *__restrict__ active, const int32_t *__restrict__ n_active, int k, int64_t H,
    int64_t I, int64_t tb0, float *__restrict__ h, uint32_t *__restrict__ hmax,
    const int32_t *__restrict__ slot_of) {
  extern __shared__ __align__(128) uint8_t ring_all[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  uint8_t *ring = ring_all + wid * (kRing * kStageBytes);
  pdl_wait();     // routing, x16 and the cleared maxima come from the previous kernel
  pdl_trigger();
  const int ipe = (int)(I / 8);
  const int nkb = (int)(H / 128);
  const int nst = (nkb + kStageKB - 1) / kStageKB;
  const int srow = (int)(2 * I / 128);
  int it_lo, it_hi;
  warp_items(*n_active * ipe, &it_lo, &it_hi);
  if (it_lo >= it_hi) return;

  // ---- producer cursor (stage being copied next)
  const CopyLane cl = copy_lane(lane);
  int is_item = it_lo, is_st = 0, is_slot = 0;
  const uint8_t *is_gate = nullptr;
  auto issue_item = [&]() {
    const int e = active[is_item / ipe];
    const int64_t ws = slot_of ? __ldg(slot_of + e) : e;  // weight slab of the expert
    const int64_t i0 = (int64_t)(is_item % ipe) * 8;
    is_gate = w13 + (ws * 2 * I + i0 + cl.rpar) * H + cl.col * 16;
  };
  issue_item();
  const int64_t up_off = I * H, two_rows = 2 * H;
  auto issue = [&]() {
    if (is_item < it_hi) {
      const int kb0 = is_st * kStageKB;
      if (kb0 + 1 < nkb || cl.col < 8) {
        uint8_t *dst = ring + is_slot * kStageBytes + cl.soff;
        const uint8_t *src = is_gate + kb0 * 128;
#pragma unroll
        for (int m = 0; m < 4; ++m) cp_async16(dst + m * 256, src + m * two_rows);
#pragma unroll
        for (int m = 0; m < 4; ++m) cp_async16(dst + (m + 4) * 256, src + up_off + m * two_rows);
      }
      if (++is_slot == kRing) is_slot = 0;
      if (++is_st == nst) {
        is_st = 0;
        if (++is_item < it_hi) issue_item();
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int st = 0; st < kRing - 1; ++st) issue();

  // ---- consumer
  const int f0 = stage_off(0, g, q), f1 = stage_off(0, g, 4 + q);  // rows g; rows g + 8 at +1024
  float tot[NT][4];
  int64_t cnt = 0, seg = 0, i0 = 0;
  const float *sg = nullptr, *su = nullptr;
  const __half *xrow[NT];
  uint4 xn[4];
  int slot = 0;
  for (int item = it_lo; item < it_hi; ++item) {
    {
      const int e = active[item / ipe];
      i0 = (int64_t)(item % ipe) * 8;
      cnt = counts[e] - tb0;
      seg = offsets[e] + tb0;
      sg = s13 + ((int64_t)e * srow + i0 / 128) * nkb;
      su = s13 + ((int64_t)e * srow + (I + i0) / 128) * nkb;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int64_t ti = j * 8 + g;
        xrow[j] = (ti < cnt) ? x16 + (int64_t)(perm[seg + ti] / k) * H + q * 16 : nullptr;
#pragma unroll
        for (int v = 0; v < 4; ++v) tot[j][v] = 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        xn[u] = xrow[0] ? ld_ro16(xrow[0] + (u >> 1) * 64 + (u & 1) * 8) : make_uint4(0, 0, 0, 0);
    }
    for (int st = 0; st < nst; ++st) {
      __syncwarp();  // every lane is done reading the slot that is refilled next
      issue();
      cp_async_wait<kRing - 1>();
      __syncwarp();
      const uint8_t *sw = ring + slot * kStageBytes;
      if (++slot == kRing) slot = 0;
      const int kb0 = st * kStageKB;
      const int nkbl = (nkb - kb0) < kStageKB ? (nkb - kb0) : kStageKB;
      for (int kbl = 0; kbl < nkbl; ++kbl) {
        const int kb = kb0 + kbl;
        const float scg = __ldg(sg + kb), scu = __ldg(su + kb);
        uint4 x0[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) x0[u] = xn[u];
        if (kb + 1 < nkb && xrow[0] != nullptr) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            xn[u] = ld_ro16(xrow[0] + (kb + 1) * 128 + (u >> 1) * 64 + (u & 1) * 8);
        }
        uint32_t a[2][4][4];
        stage_fragments(sw + kbl * 2048, f0, f1, a);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          if (j * 8 >= cnt) break;
          uint4 xc[4];
          if (j == 0) {
#pragma unroll
            for (int u = 0; u < 4; ++u) xc[u] = x0[u];
          } else if (xrow[j] != nullptr) {
#pragma unroll
            for (int u = 0; u < 4; ++u) xc[u] = ld_ro16(xrow[j] + kb * 128 + (u >> 1) * 64 + (u & 1) * 8);
          } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) xc[u] = make_uint4(0, 0, 0, 0);
          }
          float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};  // two MMA chains
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4)
#pragma unroll
            for (int c = 0; c < 2; ++c)
              mma_16816(acc[c], a[c][s4][0], a[c][s4][1], a[c][s4][2], a[c][s4][3],
                        u4_word(xc[2 * c + (s4 >> 1)], (2 * s4) & 3),
                        u4_word(xc[2 * c + (s4 >> 1)], (2 * s4 + 1) & 3));
          tot[j][0] = fmaf(acc[0][0] + acc[1][0], scg, tot[j][0]);
          tot[j][1] = fmaf(acc[0][1] + acc[1][1], scg, tot[j][1]);
          tot[j][2] = fmaf(acc[0][2] + acc[1][2], scu, tot[j][2]);
          tot[j][3] = fmaf(acc[0][3] + acc[1][3], scu, tot[j][3]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int d = 0; d < 2; ++d) {
        const int64_t ti = j * 8 + 2 * q + d;
        if (ti >= cnt) continue;
        const int64_t pos = seg + ti;
        const float xs = xscale[perm[pos] / k];
        const float hv = swiglu(tot[j][d] * xs, tot[j][2 + d] * xs);
        h[pos * I + i0 + g] = hv;
        atomicMax(&hmax[pos], __float_as_uint(fabsf(hv)));
      }
    }
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------- W2
// Item = (active expert, 16 consecutive output rows j0..j0+15), one warp, all
// of K = I.  The activations h (f32, read through L1) are split into an f16
// pair hi + lo after an exact power-of-two scaling chosen from the position's
// largest |h|, so the products keep about 22 bits of h.
template <int NT>
__global__ void __launch_bounds__(32 * kGemvWarps) gemv2_kernel(
    const uint8_t *__restrict__ w2, const float *__restrict__ s2, const float *__restrict__ h,
    const uint32_t *__restrict__ hmax, const int32_t *__restrict__ counts,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ active,
    const int32_t *__restrict__ n_active, int64_t H, int64_t I, int64_t tb0,
    float *__restrict__ y, const int32_t *__restrict__ slot_of) {
  extern __shared__ __align__(128) uint8_t ring_all[];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  uint8_t *ring = ring_all + wid * (kRing * kStageBytes);
  const int ipe = (int)(H / 16);
  const int nkb = (int)(I / 128);
  const int nst = (nkb + kStageKB - 1) / kStageKB;
  int it_lo, it_hi;
  warp_items(*n_active * ipe, &it_lo, &it_hi);
  if (it_lo >= it_hi) return;

  const CopyLane cl = copy_lane(lane);
  int is_item = it_lo, is_st = 0, is_slot = 0;
  const uint8_t *is_row = nullptr;
  auto issue_item = [&]() {
    const int e = active[is_item / ipe];
    const int64_t ws = slot_of ? __ldg(slot_of + e) : e;  // weight slab of the expert
    const int64_t j0 = (int64_t)(is_item % ipe) * 16;
    is_row = w2 + (ws * H + j0 + cl.rpar) * I + cl.col * 16;
  };
  issue_item();
  const int64_t two_rows = 2 * I;
  auto issue = [&]() {
    if (is_item < it_hi) {
      const int kb0 = is_st * kStageKB;
      if (kb0 + 1 < nkb || cl.col < 8) {
        uint8_t *dst = ring + is_slot * kStageBytes + cl.soff;
        const uint8_t *src = is_row + kb0 * 128;
#pragma unroll
        for (int m = 0; m < 8; ++m) cp_async16(dst + m * 256, src + m * two_rows);
      }
      if (++is_slot == kRing) is_slot = 0;
      if (++is_st == nst) {
        is_st = 0;
        if (++is_item < it_hi) issue_item();
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int st = 0; st < kRing - 1; ++st) issue();
  // the routing was complete before the previous kernel started; h and its
  // maxima are that kernel's output
  pdl_wait();
  pdl_trigger();

  const int f0 = stage_off(0, g, q), f1 = stage_off(0, g, 4 + q);
  float tot[NT][4];
  int64_t j0 = 0, cnt = 0, seg = 0;
  const float *sc = nullptr;
  const float *hrow[NT];
  float down[NT];
  int slot = 0;
  for (int item = it_lo; item < it_hi; ++item) {
    {
      const int e = active[item / ipe];
      j0 = (int64_t)(item % ipe) * 16;
      cnt = counts[e] - tb0;
      seg = offsets[e] + tb0;
      sc = s2 + ((int64_t)e * (H / 128) + j0 / 128) * nkb;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int64_t ti = j * 8 + g;
        hrow[j] = (ti < cnt) ? h + (seg + ti) * I + q * 16 : nullptr;
        down[j] = (ti < cnt) ? exp2i(-f16_range_shift(__uint_as_float(hmax[seg + ti]))) : 0.f;
#pragma unroll
        for (int v = 0; v < 4; ++v) tot[j][v] = 0.f;
      }
    }
    for (int st = 0; st < nst; ++st) {
      __syncwarp();
      issue();
      cp_async_wait<kRing - 1>();
      __syncwarp();
      const uint8_t *sw = ring + slot * kStageBytes;
      if (++slot == kRing) slot = 0;
      const int kb0 = st * kStageKB;
      const int nkbl = (nkb - kb0) < kStageKB ? (nkb - kb0) : kStageKB;
      for (int kbl = 0; kbl < nkbl; ++kbl) {
        const int kb = kb0 + kbl;
        const float sck = __ldg(sc + kb);
        uint32_t a[2][4][4];
        stage_fragments(sw + kbl * 2048, f0, f1, a);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          if (j * 8 >= cnt) break;
          float acc[4] = {0.f, 0.f, 0.f, 0.f}, acl[4] = {0.f, 0.f, 0.f, 0.f};  // hi and lo chains
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t bhi[8], blo[8];
            if (hrow[j] != nullptr) {
              const float4 *src = reinterpret_cast<const float4 *>(hrow[j] + kb * 128 + c * 64);
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                float4 v = __ldg(src + m);
                v.x *= down[j]; v.y *= down[j]; v.z *= down[j]; v.w *= down[j];
                const uint32_t h0 = pack_f16x2(v.x, v.y), h1 = pack_f16x2(v.z, v.w);
                const float2 r0 = unpack_f16x2(h0), r1 = unpack_f16x2(h1);
                bhi[2 * m] = h0;
                bhi[2 * m + 1] = h1;
                blo[2 * m] = pack_f16x2(v.x - r0.x, v.y - r0.y);
                blo[2 * m + 1] = pack_f16x2(v.z - r1.x, v.w - r1.y);
              }
            } else {
#pragma unroll
              for (int m = 0; m < 8; ++m) { bhi[m] = 0u; blo[m] = 0u; }
            }
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
              mma_16816(acc, a[c][s4][0], a[c][s4][1], a[c][s4][2], a[c][s4][3], bhi[2 * s4], bhi[2 * s4 + 1]);
              mma_16816(acl, a[c][s4][0], a[c][s4][1], a[c][s4][2], a[c][s4][3], blo[2 * s4], blo[2 * s4 + 1]);
            }
          }
#pragma unroll
          for (int v = 0; v < 4; ++v) tot[j][v] = fmaf(acc[v] + acl[v], sck, tot[j][v]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int d = 0; d < 2; ++d) {
        const int64_t ti = j * 8 + 2 * q + d;
        if (ti >= cnt) continue;
        const int64_t pos = seg + ti;
        const float up = exp2i(f16_range_shift(__uint_as_float(hmax[pos])));
        y[pos * H + j0 + g] = tot[j][d] * up;
        y[pos * H + j0 + 8 + g] = tot[j][2 + d] * up;
      }
    }
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------- combine
// out[t, :] = bf16_rne( sum_{r=0}^{k-1} w[t, r] * y[inv[t k + r], :] ), summed
// in router rank order with one fma chain per element (WARP BACKENDS.md,
// "Coherent memory": partials reduced in original router order) and no atomics.
// y of a pair is the sum of its rows in NP planes, added in plane order.
// Thread: one 4-column group of one token; the loads of up to kCombineBatch
// pairs (all planes) are issued before any is used.
constexpr int kCombineThreads = 64;
constexpr int kCombineBatch = 8;

template <int NP>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const float *__restrict__ y, int64_t plane,
                                                                  const int32_t *__restrict__ inv,
                                                                  const float *__restrict__ wts, int64_t T,
                                                                  int k, int64_t H,
                                                                  __nv_bfloat16 *__restrict__ out) {
  const int64_t t = blockIdx.x;
  const int64_t j = 4 * ((int64_t)blockIdx.y * kCombineThreads + threadIdx.x);
  pdl_wait();
  if (t >= T || j >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r0 = 0; r0 < k; r0 += kCombineBatch) {
    float4 v[kCombineBatch][NP];
    float w[kCombineBatch];
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      if (r0 + u < k) {
        const int64_t pos = __ldg(inv + t * k + r0 + u);
        w[u] = __ldg(wts + t * k + r0 + u);
#pragma unroll
        for (int q = 0; q < NP; ++q) v[u][q] = __ldg(reinterpret_cast<const float4 *>(y + q * plane + pos * H + j));
      }
    }
#pragma unroll
    for (int u = 0; u < kCombineBatch; ++u) {
      if (r0 + u < k) {
        float4 s4 = v[u][0];
#pragma unroll
        for (int q = 1; q < NP; ++q) {
          s4.x += v[u][q].x;
          s4.y += v[u][q].y;
          s4.z += v[u][q].z;
          s4.w += v[u][q].w;
        }
        acc.x = fmaf(w[u], s4.x, acc.x);
        acc.y = fmaf(w[u], s4.y, acc.y);
        acc.z = fmaf(w[u], s4.z, acc.z);
        acc.w = fmaf(w[u], s4.w, acc.w);
      }
    }
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 o;
  o.x = *reinterpret_cast<uint32_t *>(&lo);
  o.y = *reinterpret_cast<uint32_t *>(&hi);
  *reinterpret_cast<uint2 *>(out + t * H + j) = o;
}

// ---------------------------------------------------------------- launchers

namespace {
template <typename K>
cudaError_t allow_smem(K kernel, size_t smem) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}
constexpr size_t kGemvSmem = (size_t)kGemvWarps * kRing * kStageBytes;
// grid: enough warps for every item, but never more CTAs than fit on the GPU
// at once (each warp owns a fixed item range, so a second wave would run late)
template <typename K>
int64_t gemv_grid(K kernel, int64_t max_items, int sms) {
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 32 * kGemvWarps, kGemvSmem) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t g = (max_items + kGemvWarps - 1) / kGemvWarps;
  const int64_t cap = (int64_t)sms * per_sm;
  return g < cap ? g : cap;
}
}  // namespace

// Token groups of up to 8 * NT per pass; T <= 8 needs one group (NT = 1),
// T <= 64 fits in NT = 8; larger T runs ceil(T / 64) passes of 64 tokens.
cudaError_t launch_gemv13(const uint8_t *w13, const float *s13, const __half *x16,
                          const float *xscale, const int32_t *counts, const int32_t *offsets,
                          const int32_t *perm, const int32_t *active, const int32_t *n_active,
                          int k, int64_t T, int64_t H, int64_t I, float *h, uint32_t *hmax,
                          int64_t max_items, int *err, int sms, cudaStream_t s,
                          const int32_t *slot_of) {
  cudaError_t e;
  if (T <= 8) {
    auto kern = gemv13_swiglu_kernel<1>;
    if ((e = allow_smem(kern, kGemvSmem)) != cudaSuccess) return e;
    const int64_t grid = gemv_grid(kern, max_items, sms);
    if (grid <= 0) return cudaSuccess;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(32 * kGemvWarps), kGemvSmem, s, w13, s13, x16,
                      xscale, counts, offsets, perm, active, n_active, k, H, I, (int64_t)0, h, hmax,
                      slot_of);
  }
  auto kern = gemv13_swiglu_kernel<8>;
  if ((e = allow_smem(kern, kGemvSmem)) != cudaSuccess) return e;
  const int64_t grid = gemv_grid(kern, max_items, sms);
  if (grid <= 0) return cudaSuccess;
  for (int64_t tb0 = 0; tb0 < T; tb0 += 64)
    kern<<<(unsigned)grid, 32 * kGemvWarps, kGemvSmem, s>>>(w13, s13, x16, xscale, counts, offsets,
                                                            perm, active, n_active, k, H, I, tb0, h,
                                                            hmax, slot_of);
  return cudaGetLastError();
}

cudaError_t launch_gemv2(const uint8_t *w2, const float *s2, const float *h, const uint32_t *hmax,
                         const int32_t *counts, const int32_t *offsets, const int32_t *active,
                         const int32_t *n_active, int64_t T, int64_t H, int64_t I, float *y,
                         int64_t max_items, int *err, int sms, cudaStream_t s,
                         const int32_t *slot_of) {
  cudaError_t e;
  if (T <= 8) {
    auto kern = gemv2_kernel<1>;
    if ((e = allow_smem(kern, kGemvSmem)) != cudaSuccess) return e;
    const int64_t grid = gemv_grid(kern, max_items, sms);
    if (grid <= 0) return cudaSuccess;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(32 * kGemvWarps), kGemvSmem, s, w2, s2, h, hmax,
                      counts, offsets, active, n_active, H, I, (int64_t)0, y, slot_of);
  }
  auto kern = gemv2_kernel<8>;
  if ((e = allow_smem(kern, kGemvSmem)) != cudaSuccess) return e;
  const int64_t grid = gemv_grid(kern, max_items, sms);
  if (grid <= 0) return cudaSuccess;
  for (int64_t tb0 = 0; tb0 < T; tb0 += 64)
    kern<<<(unsigned)grid, 32 * kGemvWarps, kGemvSmem, s>>>(w2, s2, h, hmax, counts, offsets,
                                                            active, n_active, H, I, tb0, y, slot_of);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float *y, int n_planes, int64_t plane, const int32_t *inv,
                           const float *wts, int64_t T, int k, int64_t H, __nv_bfloat16 *out,
                           cudaStream_t s) {
  const dim3 grid((unsigned)T, (unsigned)((H / 4 + kCombineThreads - 1) / kCombineThreads));
  if (n_planes == 3)
    return launch_pdl(combine_kernel<3>, grid, dim3(kCombineThreads), 0, s, y, plane, inv, wts, T, k, H, out);
  if (n_planes != 1) return cudaErrorInvalidValue;
  return launch_pdl(combine_kernel<1>, grid, dim3(kCombineThreads), 0, s, y, plane, inv, wts, T, k, H, out);
}

}  // namespace fp8moe
