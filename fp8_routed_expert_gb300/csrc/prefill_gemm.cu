// Grouped FP8 GEMM of the routed experts for large batches (prefill), on the
// 5th-generation tensor cores (tcgen05 + TMEM) fed by TMA.
//
// The whole prompt goes through the layer at once and each expert's rows are
// processed as one GEMM over its token segment (DeepSeek-V4.1-Flash post, §5
// "Don't read 66 GB per prompt chunk"), so every expert weight tile is read
// from HBM once per batch rather than once per token.
//
// Operands.  B is the expert weight (e4m3 codes, one f32 scale per 128x128
// block).  A is the permuted activation rows, split per (row, 128-column
// block) into NT e4m3 terms that share one power-of-two scale 2^e (the
// smallest with amax / 2^e <= 448): x / 2^e ~= t0 + t1 (+ t2).  One e4m3 term
// alone is 4e-2 away from the exact layer in relative L2 (the pages count
// 8-bit activations as an accuracy change: Trochilus "Results", WARP
// BACKENDS.md int8 activation table).  Each term carries 4 significant bits:
// two terms hold a bf16 activation exactly, so GEMM1 (x is bf16) uses two;
// GEMM2's input h is an f32 intermediate and gets three (about 12 bits).
// All terms are multiplied against the same B tile into one TMEM accumulator.
//
// Block-scale promotion.  For every 128-wide K block the MMA warp accumulates
// into one of two TMEM buffers (128 lanes x 256 f32 columns each); the
// epilogue warps read that partial and add partial * s_a[row, kb] * s_w[block,
// kb] to f32 registers, while the MMA warp fills the other buffer.  This is
// the per-128-column scale folding of dragon.c §8 "Round 3", done per K block
// in f32.
//
// Tile: 128 rows (positions of one expert's segment) x 256 columns x K.  A
// tile with at most 64 rows in the segment (most experts of a large, skewed
// batch hold only a few dozen positions) loads 64 activation rows and runs
// M = 64 MMAs, half the tensor work; its accumulator rows then sit in TMEM
// lanes 32 q + l, l < 16 (row 16 q + l), so each epilogue warp holds 16 rows.
//   GEMM1 (gate/up): the 256 B rows are gate rows [n0, n0+64), up rows
//   [I+n0, I+n0+64), gate rows [n0+64, n0+128), up rows [I+n0+64, I+n0+128)
//   with n0 = 128 nb, so each epilogue warp holds the gate and up values of
//   the same h outputs and applies SwiGLU itself; the 128 h values of a row
//   block are then split into three e4m3 terms with one power-of-two scale
//   (the A operand of GEMM2).
//   GEMM2 (down): 256 consecutive rows of W2; the epilogue stores f32 y.
// Warp roles (320 threads, one CTA per SM, persistent over work items
// (expert tile, column block)): warp 0 issues TMA, warp 1 allocates TMEM and
// issues tcgen05.mma, warps 2..9 promote and finish the tile.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace fp8moe {
using namespace sm100;

namespace {

constexpr int BM = 128, BN = 256, BK = 128;
constexpr int A_TILE = BM * BK;                    // bytes of one e4m3 term
constexpr int B_TILE = BN * BK;
constexpr int B_BOX_ROWS = 64;
constexpr int NUM_EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s per wait

// Output staging per epilogue warp: the boxes its 32 rows send to global
// memory by TMA store (gate/up: 3 h terms x 32 rows x 32 bytes per round;
// down: two 32 x 32 f32 boxes).
template <int NT>
struct Pipe {
  static constexpr int STAGE_BYTES = NT * A_TILE + B_TILE;  // 64 KiB (NT=2) or 80 KiB (NT=3)
  static constexpr int STAGES = NT == 2 ? 3 : 2;
  static constexpr int STG_WARP = NT == 2 ? 4096 : 8192;
  static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + (size_t)NUM_EPI_WARPS * STG_WARP + 1024;
};

struct GemmArgs {
  const int32_t *offsets;       // [E+1]
  const int32_t *tile_offsets;  // [E+1] exclusive scan of ceil(count / 128)
  const float *a_scale;         // [K/128][Pmax]
  const float *w_scale;         // s13 [E][2I/128][H/128] or s2 [E][H/128][I/128]
  int E;
  int64_t K;                    // reduction length: H (GEMM1) or I (GEMM2)
  int64_t H, I, Pmax;
  int64_t n_blocks;             // GEMM1: I/128, GEMM2: H/256
  uint8_t *h_t0, *h_t1, *h_t2;  // GEMM1 outputs: three e4m3 terms [Pmax, I]
  float *h_scale;               //               power-of-two scales [I/128][Pmax]
  float *y;                     // GEMM2 output [Pmax, H]
  int *err;
  const int32_t *slot_of;       // weight slab of each expert, or nullptr (slab = expert)
};

struct ItemCoords {
  int e, nb;
  int64_t m0, row_end;
};

__device__ __forceinline__ ItemCoords item_coords(const GemmArgs &p, int64_t item) {
  ItemCoords c;
  const int64_t ti = item / p.n_blocks;
  c.nb = (int)(item % p.n_blocks);
  int lo = 0, hi = p.E;  // largest e with tile_offsets[e] <= ti
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.tile_offsets[mid] <= ti) lo = mid;
    else hi = mid;
  }
  c.e = lo;
  c.m0 = p.offsets[lo] + (ti - p.tile_offsets[lo]) * BM;
  c.row_end = p.offsets[lo + 1];
  return c;
}

__device__ __forceinline__ void raise_abort(volatile int *abort_flag, int *err) {
  *abort_flag = 1;
  set_error(err, DEV_ERR_TIMEOUT);
}

template <int MODE, int NT>
__global__ void __launch_bounds__(THREADS, 1) grouped_gemm_kernel(const __grid_constant__ TmapSet tm,
                                                                 const GemmArgs p) {
  constexpr int STAGES = Pipe<NT>::STAGES, STAGE_BYTES = Pipe<NT>::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES], tfull_bar[2], tempty_bar[2];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;
  __shared__ float amax_x[2][BM];

  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nkb = p.K / BK;
  const int64_t n_items = (int64_t)p.tile_offsets[p.E] * p.n_blocks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], NUM_EPI_WARPS);
    }
    abort_flag = 0;
    fence_mbar_init();
    for (int t = 0; t < NT; ++t) {
      prefetch_tmap(&tm.a[t]);
      prefetch_tmap(&tm.a64[t]);
    }
    prefetch_tmap(&tm.b);
    for (int t = 0; t < (MODE == 1 ? 3 : 1); ++t) prefetch_tmap(&tm.st[t]);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int64_t item = blockIdx.x; item < n_items && !abort_flag; item += gridDim.x) {
        const ItemCoords c = item_coords(p, item);
        int64_t b_rows[4];
        const int64_t ws = p.slot_of ? __ldg(p.slot_of + c.e) : c.e;  // weight slab
        if (MODE == 1) {
          const int64_t g = ws * 2 * p.I + (int64_t)c.nb * 128;
          const int64_t u = g + p.I;
          b_rows[0] = g; b_rows[1] = u; b_rows[2] = g + 64; b_rows[3] = u + 64;
        } else {
          const int64_t r = ws * p.H + (int64_t)c.nb * 256;
          b_rows[0] = r; b_rows[1] = r + 64; b_rows[2] = r + 128; b_rows[3] = r + 192;
        }
        const bool half_m = c.row_end - c.m0 <= 64;  // M = 64 item: 64 activation rows
        for (int64_t kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, &abort_flag, WAIT_LIMIT_NS)) {
            raise_abort(&abort_flag, p.err);
            break;
          }
          uint8_t *sa = smem + (size_t)stage * STAGE_BYTES;
          mbar_arrive_expect_tx(&full_bar[stage], STAGE_BYTES - (half_m ? NT * A_TILE / 2 : 0));
          const int32_t kx = (int32_t)(kb * BK);
#pragma unroll
          for (int t = 0; t < NT; ++t)
            tma_load_2d(sa + t * A_TILE, half_m ? &tm.a64[t] : &tm.a[t], kx, (int32_t)c.m0,
                        &full_bar[stage]);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            tma_load_2d(sa + NT * A_TILE + q * (B_BOX_ROWS * BK), &tm.b, kx, (int32_t)b_rows[q],
                        &full_bar[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc128 = idesc_e4m3_f32(BM, BN), idesc64 = idesc_e4m3_f32(64, BN);
      int stage = 0, buf = 0;
      uint32_t phase = 0, bphase = 0;
      for (int64_t item = blockIdx.x; item < n_items && !abort_flag; item += gridDim.x) {
        const ItemCoords c = item_coords(p, item);
        const uint32_t idesc = c.row_end - c.m0 <= 64 ? idesc64 : idesc128;
        for (int64_t kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&tempty_bar[buf], bphase ^ 1u, &abort_flag, WAIT_LIMIT_NS) ||
              !mbar_wait(&full_bar[stage], phase, &abort_flag, WAIT_LIMIT_NS)) {
            raise_abort(&abort_flag, p.err);
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + (size_t)stage * STAGE_BYTES);
          const uint32_t b = a0 + NT * A_TILE;
          const uint32_t d = tmem + (uint32_t)buf * BN;
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            const uint64_t bd = sw128_kmajor_desc(b + kk * 32);
#pragma unroll
            for (int t = 0; t < NT; ++t)
              mma_f8f6f4(d, sw128_kmajor_desc(a0 + t * A_TILE + kk * 32), bd, idesc,
                         (kk > 0 || t > 0) ? 1u : 0u);
          }
          mma_commit(&empty_bar[stage]);
          mma_commit(&tfull_bar[buf]);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          buf ^= 1;
          if (buf == 0) bphase ^= 1u;
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- promotion + epilogue
    const int quarter = warp & 3;             // TMEM lanes this warp may read
    const int half = (warp - 2) >> 2;         // column half of the 256-wide tile
    uint8_t *stg_warp = smem + (size_t)STAGES * STAGE_BYTES + (size_t)(warp - 2) * Pipe<NT>::STG_WARP;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    int buf = 0;
    uint32_t bphase = 0;
    const int64_t wrow_blocks = (MODE == 1) ? 2 * p.I / 128 : p.H / 128;
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
      ItemCoords c = item_coords(p, item);
      // rows per warp: 32 (M = 128 item) or 16 (M = 64: lanes 16..31 idle)
      const int rpw = c.row_end - c.m0 <= 64 ? 16 : 32;
      const bool lane_ok = lane < rpw;
      const int r_in_tile = quarter * rpw + lane;
      const int64_t row = c.m0 + r_in_tile;
      // weight scales of the two 128-row blocks of this tile half: gate and up
      // rows (GEMM1) or one W2 row block (GEMM2), one per K block
      const float *ws = p.w_scale + (int64_t)c.e * wrow_blocks * nkb;
      const float *ws0 = ws + (MODE == 1 ? (int64_t)c.nb : 2 * (int64_t)c.nb + half) * nkb;
      const float *ws1 = ws + (MODE == 1 ? p.I / 128 + c.nb : 2 * (int64_t)c.nb + half) * nkb;
      float acc[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0.f;
      bool ok = true;
      const bool sa_ok = lane_ok && row < p.Pmax;
      const float *sa_p = p.a_scale + (sa_ok ? row : 0);
      // the scales of K block kb + 1 are loaded while block kb is promoted,
      // so their latency is not on the path between the MMA and the epilogue
      float sa_n = sa_ok ? __ldg(sa_p) : 0.f;
      float s0_n = __ldg(ws0), s1_n = __ldg(ws1);
      const int nkb32 = (int)nkb;
      for (int kb = 0; kb < nkb32; ++kb) {
        const float c0 = sa_n * s0_n, c1 = sa_n * s1_n;
        if (kb + 1 < nkb32) {
          sa_p += p.Pmax;
          sa_n = sa_ok ? __ldg(sa_p) : 0.f;
          s0_n = __ldg(ws0 + kb + 1);
          s1_n = __ldg(ws1 + kb + 1);
        }
        // no early exit on the abort flag here: the epilogue warps share a
        // named barrier, so they must all stop at the same (timed-out) wait
        if (!mbar_wait(&tfull_bar[buf], bphase, nullptr, WAIT_LIMIT_NS)) {
          raise_abort(&abort_flag, p.err);
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          float v[16];
          tmem_ld_32x32b_x16(t_lane + (uint32_t)(buf * BN + half * 128 + ch * 16), v);
          const float sc = ch < 4 ? c0 : c1;
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[ch * 16 + j] = fmaf(v[j], sc, acc[ch * 16 + j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty_bar[buf]);
        buf ^= 1;
        if (buf == 0) bphase ^= 1u;
      }
      if (!ok) break;
      // the item's coordinates again, rather than keeping them in registers
      // through the K loop
      c = item_coords(p, item);
      const bool valid = lane_ok && row < c.row_end;

      if (MODE == 1) {
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          acc[j] = valid ? swiglu(acc[j], acc[64 + j]) : 0.f;  // rows past the segment hold garbage
          amax = fmaxf(amax, fabsf(acc[j]));
        }
        if (lane_ok) amax_x[half][r_in_tile] = amax;
        named_bar_sync(1, 32 * NUM_EPI_WARPS);
        const float am = lane_ok ? fmaxf(amax_x[0][r_in_tile], amax_x[1][r_in_tile]) : 0.f;
        named_bar_sync(1, 32 * NUM_EPI_WARPS);
        // The warp's 32 rows go out through its staging buffer: whole boxes
        // by TMA store (asynchronous) when all 32 rows lie in the segment,
        // else the valid rows by plain 16-byte copies from the buffer.
        const int ex = e4m3_block_exponent(am);
        const Pow2 down = pow2_factors(-ex);
        const int32_t x0 = (int32_t)(c.nb * 128 + half * 64), y0 = (int32_t)(c.m0 + quarter * rpw);
        int64_t nrows = c.row_end - y0;  // rows of this warp in the segment (may be <= 0)
        if (nrows > rpw) nrows = rpw;
        const bool full_q = nrows == 32;  // warp-uniform
        uint32_t ln;  // opaque copy of the lane index (see the down GEMM's tail)
        asm volatile("mov.u32 %0, %1;" : "=r"(ln) : "r"((uint32_t)lane));
        uint8_t *srow = stg_warp + ln * 32;
#pragma unroll
        for (int rd = 0; rd < 2; ++rd) {
          if (lane == 0) bulk_wait_read<0>();  // earlier boxes have left the buffer
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 32; j += 16) {
            uint32_t w0[4], w1[4], w2[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              uint32_t a[3], b[3];
              const int v = rd * 32 + j + 4 * m;
              e4m3_terms<3>(down(acc[v]), down(acc[v + 1]), a);
              e4m3_terms<3>(down(acc[v + 2]), down(acc[v + 3]), b);
              w0[m] = a[0] | (b[0] << 16);
              w1[m] = a[1] | (b[1] << 16);
              w2[m] = a[2] | (b[2] << 16);
            }
            *reinterpret_cast<uint4 *>(srow + 0 * 1024 + j) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
            *reinterpret_cast<uint4 *>(srow + 1 * 1024 + j) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
            *reinterpret_cast<uint4 *>(srow + 2 * 1024 + j) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
          }
          if (full_q) {
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tm.st[0], stg_warp, x0 + rd * 32, y0);
              tma_store_2d(&tm.st[1], stg_warp + 1024, x0 + rd * 32, y0);
              tma_store_2d(&tm.st[2], stg_warp + 2048, x0 + rd * 32, y0);
              bulk_commit();
            }
          } else if (nrows > 0) {
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 6; ++i) {  // 3 terms x 32 rows x two 16-byte pieces
              const int idx = i * 32 + lane, t = idx >> 6, r = (idx >> 1) & 31, pc = idx & 1;
              if (r < nrows) {
                uint8_t *dst = (t == 0 ? p.h_t0 : t == 1 ? p.h_t1 : p.h_t2) +
                               (int64_t)(y0 + r) * p.I + x0 + rd * 32 + pc * 16;
                *reinterpret_cast<uint4 *>(dst) =
                    *reinterpret_cast<const uint4 *>(stg_warp + t * 1024 + r * 32 + pc * 16);
              }
            }
            __syncwarp();
          }
        }
        if (valid && half == 0) p.h_scale[(int64_t)c.nb * p.Pmax + row] = ldexpf(1.f, ex);
      } else {
        // four 32 x 32 f32 boxes through two 128-byte-swizzled buffers (16-byte
        // piece q of row r sits at piece q ^ (r % 8)): TMA stores when all 32
        // rows of the warp lie in the segment, else plain copies of the valid rows
        const int32_t y0 = (int32_t)(c.m0 + quarter * rpw);
        int64_t nrows = c.row_end - y0;
        if (nrows > rpw) nrows = rpw;
        const bool full_q = nrows == 32;  // warp-uniform
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint8_t *b = stg_warp + (ch & 1) * 4096;
          const int32_t x = (int32_t)(c.nb * 256 + half * 128 + ch * 32);
          if (ch >= 2) {
            if (lane == 0) bulk_wait_read<1>();  // the box of chunk ch - 2 has left b
            __syncwarp();
          }
          // the row's base address is formed here (an opaque copy of the lane
          // index), so the compiler does not keep eight swizzled addresses
          // live through the K loop
          uint32_t ln;
          asm volatile("mov.u32 %0, %1;" : "=r"(ln) : "r"((uint32_t)lane));
          uint8_t *brow = b + ln * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4 *>(brow + ((q ^ (ln & 7)) << 4)) =
                make_float4(acc[ch * 32 + 4 * q], acc[ch * 32 + 4 * q + 1], acc[ch * 32 + 4 * q + 2],
                            acc[ch * 32 + 4 * q + 3]);
          if (full_q) {
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tm.st[0], b, x, y0);
              bulk_commit();
            }
          } else if (nrows > 0) {
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {  // 32 rows x eight 16-byte pieces
              const int idx = i * 32 + lane, r = idx >> 3, q = idx & 7;
              if (r < nrows)
                *reinterpret_cast<float4 *>(p.y + (int64_t)(y0 + r) * p.H + x + q * 4) =
                    *reinterpret_cast<const float4 *>(b + r * 128 + ((q ^ (r & 7)) << 4));
            }
            __syncwarp();
          }
        }
      }
    }
    if (lane == 0) bulk_wait<0>();  // every TMA store of this warp has completed
    __syncwarp();
  }

  __syncthreads();
  if (abort_flag) {
    // let copies and MMAs already in flight land before the memory goes away
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 50000ull) {
    }
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- activation quantisation
// One bf16 row of H columns -> two e4m3 terms per 128-column block sharing
// the block's power-of-two scale (a bf16 value is held exactly by the two
// terms).  One warp per row: lane l takes 8 consecutive columns of every
// 256-column span, so a half-warp covers one block (its amax is a 16-lane
// reduction) and four spans' 16-byte loads are in flight at once.
__device__ __forceinline__ void quant_row_2terms(const __nv_bfloat16 *__restrict__ src, int64_t H,
                                                 uint8_t *__restrict__ dhi, uint8_t *__restrict__ dlo,
                                                 float *__restrict__ scale, int64_t ld) {
  const int lane = threadIdx.x & 31;
  const int64_t nsp = (H + 255) / 256;
  for (int64_t sp0 = 0; sp0 < nsp; sp0 += 4) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t col = (sp0 + u) * 256 + lane * 8;
      v[u] = (sp0 + u < nsp && col < H) ? __ldg(reinterpret_cast<const uint4 *>(src + col))
                                        : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (sp0 + u >= nsp) break;  // uniform over the warp
      const int64_t col = (sp0 + u) * 256 + lane * 8;
      float f[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w = u4_word(v[u], i);
        f[2 * i] = bf16_bits_to_float(w & 0xffffu);
        f[2 * i + 1] = bf16_bits_to_float(w >> 16);
      }
      float am = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(f[i]));
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      const int ex = e4m3_block_exponent(am);
      const Pow2 down = pow2_factors(-ex);
      uint32_t hi[2], lo[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        uint32_t a[2], b[2];
        e4m3_terms<2>(down(f[4 * i]), down(f[4 * i + 1]), a);
        e4m3_terms<2>(down(f[4 * i + 2]), down(f[4 * i + 3]), b);
        hi[i] = a[0] | (b[0] << 16);
        lo[i] = a[1] | (b[1] << 16);
      }
      if (col < H) {
        *reinterpret_cast<uint2 *>(dhi + col) = make_uint2(hi[0], hi[1]);
        *reinterpret_cast<uint2 *>(dlo + col) = make_uint2(lo[0], lo[1]);
        if ((lane & 15) == 0) scale[(col / 128) * ld] = ldexpf(1.f, ex);
      }
    }
  }
}

// Position rows: row pos is x of token perm[pos] / k (the expert-sorted
// operand of the grouped GEMM); scales a_scale[kb * Pmax + pos].
// (four CTAs per SM: the row loop is bound by latency, not by registers)
__global__ void __launch_bounds__(256, 4) act_quant_kernel(const __nv_bfloat16 *__restrict__ x,
                                                        const int32_t *__restrict__ perm, int64_t P,
                                                        int k, int64_t H, int64_t Pmax,
                                                        uint8_t *__restrict__ a_hi,
                                                        uint8_t *__restrict__ a_lo,
                                                        float *__restrict__ a_scale) {
  pdl_wait();
  pdl_trigger();
  for (int64_t pos = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; pos < P;
       pos += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int64_t t = __ldg(perm + pos) / k;
    quant_row_2terms(x + t * H, H, a_hi + pos * H, a_lo + pos * H, a_scale + pos, Pmax);
  }
}

// Token rows: the token-major operand of the decode FFN; scales
// a_scale[kb * a_ld + t].
__global__ void __launch_bounds__(256) act_quant_tokens_kernel(const __nv_bfloat16 *__restrict__ x,
                                                               int64_t T, int64_t H,
                                                               uint8_t *__restrict__ a_hi,
                                                               uint8_t *__restrict__ a_lo,
                                                               float *__restrict__ a_scale,
                                                               int64_t a_ld) {
  pdl_wait();
  pdl_trigger();
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T;
       t += ((int64_t)gridDim.x * blockDim.x) >> 5)
    quant_row_2terms(x + t * H, H, a_hi + t * H, a_lo + t * H, a_scale + t, a_ld);
}

// ---------------------------------------------------------------- tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

// Row-major u8 matrix [rows, cols], boxes of box_rows x 128 bytes, 128-byte swizzle.
bool encode_u8_tmap(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_h_store_tmap(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_y_store_tmap(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_act_quant(const __nv_bfloat16 *x, const int32_t *perm, int64_t P, int k,
                             int64_t H, int64_t Pmax, uint8_t *a_hi, uint8_t *a_lo, float *a_scale,
                             int sms, cudaStream_t s) {
  int64_t grid = (P + 7) / 8;  // one warp per row
  const int64_t cap = (int64_t)sms * 8;
  if (grid > cap) grid = cap;
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(act_quant_kernel, dim3((unsigned)grid), dim3(256), 0, s, x, perm, P, k, H, Pmax,
                    a_hi, a_lo, a_scale);
}

cudaError_t launch_act_quant_tokens(const __nv_bfloat16 *x, int64_t T, int64_t H, uint8_t *a_hi,
                                    uint8_t *a_lo, float *a_scale, int64_t a_ld, int sms,
                                    cudaStream_t s) {
  int64_t grid = (T + 7) / 8;  // one warp per row
  const int64_t cap = (int64_t)sms * 8;
  if (grid > cap) grid = cap;
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(act_quant_tokens_kernel, dim3((unsigned)grid), dim3(256), 0, s, x, T, H, a_hi,
                    a_lo, a_scale, a_ld);
}

cudaError_t launch_grouped_gemm(int mode, const TmapSet &tm, const int32_t *offsets,
                                const int32_t *tile_offsets, const float *a_scale,
                                const float *w_scale, int E, int64_t H, int64_t I, int64_t Pmax,
                                uint8_t *const h_terms[3], float *h_scale, float *y, int *err,
                                int64_t max_items, int sms, cudaStream_t s, const int32_t *slot_of) {
  GemmArgs p;
  p.slot_of = slot_of;
  p.offsets = offsets;
  p.tile_offsets = tile_offsets;
  p.a_scale = a_scale;
  p.w_scale = w_scale;
  p.E = E;
  p.K = mode == 1 ? H : I;
  p.H = H;
  p.I = I;
  p.Pmax = Pmax;
  p.n_blocks = mode == 1 ? I / 128 : H / 256;
  p.h_t0 = h_terms ? h_terms[0] : nullptr;
  p.h_t1 = h_terms ? h_terms[1] : nullptr;
  p.h_t2 = h_terms ? h_terms[2] : nullptr;
  p.h_scale = h_scale;
  p.y = y;
  p.err = err;
  int64_t grid = max_items < sms ? max_items : sms;
  if (grid <= 0) return cudaSuccess;
  cudaError_t e;
  if (mode == 1) {
    auto k = grouped_gemm_kernel<1, 2>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Pipe<2>::SMEM);
    if (e != cudaSuccess) return e;
    k<<<(unsigned)grid, THREADS, Pipe<2>::SMEM, s>>>(tm, p);
  } else {
    auto k = grouped_gemm_kernel<2, 3>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Pipe<3>::SMEM);
    if (e != cudaSuccess) return e;
    k<<<(unsigned)grid, THREADS, Pipe<3>::SMEM, s>>>(tm, p);
  }
  return cudaGetLastError();
}

}  // namespace fp8moe
