// Grouped GEMV of the routed experts for small batches on the 5th-generation
// tensor cores: each expert's weight rows are the MMA's M = 128 operand and
// its (at most 16 per tile) tokens the N = 16 operand, so the weights stream
// from HBM through TMA into shared memory and into tcgen05.mma without any
// per-byte instruction on the SM.  The bytes moved per token decide MoE speed
// (DeepSeek-V4.1-Flash post, "Bytes per token decide everything"); here the SM
// only promotes one 128 x 16 partial per K block.
//
// Operands: A = e4m3 weight rows (one f32 scale per 128 x 128 block); B = the
// expert's activation rows in position order, split into e4m3 terms sharing a
// power-of-two scale per (row, K block): two terms for x (exact for bf16),
// three for h.  The terms sit side by side along N (N = 32 or 48), so one MMA
// per 32-wide K slice reads each weight byte from shared memory once; the
// promotion adds the terms' columns.  Every 128-wide K block (64-wide for h,
// whose scale is per 64 columns) is accumulated in its own TMEM buffer and
// added to f32 registers as partial * s_w[row block, kb] * s_act[token, block]
// (dragon.c §8 "Round 3": the block scale is folded out of the inner product).
//
//   MODE 1 (gate/up): item = (16-token tile of expert e, h outputs i0..i0+63);
//     A rows 0..63 are gate rows i0.., rows 64..127 the up rows I + i0..; the
//     epilogue forms h = silu(gate) * up and writes it as three e4m3 terms with
//     one power-of-two scale per (position, 64 outputs).
//   MODE 2 (down): item = (16-token tile, output rows j0..j0+127); y in f32.
// Warp 0 issues the TMA loads of each stage and, with 4-byte cp.async into a
// ring of its own, the stage's scales (so they arrive with the weights instead
// of behind them); warp 1 allocates TMEM and issues the MMAs; warps 2..5
// promote and finish the item.  Every mbarrier wait is bounded.
#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace fp8moe {
using namespace sm100;

namespace {

constexpr int DM = 128;      // weight rows per item
constexpr int DN = 16;       // tokens per tile
constexpr int DK = 128;      // K per stage
constexpr int A_BYTES = DM * DK;
constexpr int B_BYTES = DN * DK;
constexpr int MAX_NBUF = 8;  // TMEM partial buffers (see DPipe)
constexpr int EPI_WARPS = 4;
constexpr int SC_SLOTS = 24;   // scale ring slots, one per stage
constexpr int SC_STRIDE = 36;  // floats per slot: 2 x 16 activation scales, 2 weight scales, pad
constexpr int kMaxE = 1024;
constexpr int DTHREADS = 64 + 32 * EPI_WARPS;
constexpr uint64_t DWAIT_NS = 2000000000ull;

template <int NT>
struct DPipe {
  static constexpr int STAGE = A_BYTES + NT * B_BYTES;  // 20 KiB (NT=2) / 22 KiB (NT=3)
  static constexpr int STAGES = 8;
  static constexpr size_t SMEM = (size_t)STAGES * STAGE + 1024;
  static constexpr int NC = NT * DN;                     // MMA N: the terms side by side
  static constexpr int BUF_COLS = NC <= 32 ? 32 : 64;    // TMEM columns per partial buffer
  // gate/up: 8 buffers, so the MMAs run on while an item's SwiGLU and
  // quantisation tail is computed; down (a short tail): 4
  static constexpr int NBUF = NT == 2 ? 8 : 4;
  static constexpr uint32_t TMEM_COLS = NBUF * BUF_COLS; // 256
};

struct DecodeArgs {
  const int32_t *offsets, *tile_offsets;  // tile offsets in units of DN-token tiles
  const float *act_scale;                 // [K/blk][Pmax], blk = 128 (x) or 64 (h)
  const float *w_scale;                   // s13 or s2
  int E;
  int64_t H, I, Pmax;
  int n_blocks;                           // MODE 1: I/64, MODE 2: H/128
  uint8_t *h_t0, *h_t1, *h_t2;            // MODE 1 outputs [Pmax, I]
  float *h_scale;                         // [I/64][Pmax]
  float *y;                               // MODE 2 output [Pmax, H]
  int *err;
};

struct DItem {
  int e, nb;
  int64_t p0, p_end;  // first position of the tile, end of the expert's segment
};

// Item -> (expert, row block, tile positions), from shared-memory copies of
// the tile and position offsets.
__device__ __forceinline__ DItem ditem(const int *toff, const int *off, int E, int n_blocks,
                                       int64_t item) {
  DItem c;
  const int64_t ti = item / n_blocks;
  c.nb = (int)(item % n_blocks);
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (toff[mid] <= ti) lo = mid;
    else hi = mid;
  }
  c.e = lo;
  c.p0 = off[lo] + (ti - toff[lo]) * DN;
  c.p_end = off[lo + 1];
  return c;
}

// 32 lanes x 16 consecutive f32 columns of TMEM (no wait).
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t *v) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}

// 4-byte asynchronous copy global -> shared, tracked by cp.async.mbarrier.arrive.
__device__ __forceinline__ void cp_async4(float *dst, const float *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// Arrive on `bar` once this thread's earlier cp.async copies have landed
// (without first raising the pending count: the barrier's count includes
// this thread).
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int MODE, int NT>
__global__ void __launch_bounds__(DTHREADS, 1) decode_mma_kernel(const __grid_constant__ TmapSet tm,
                                                                 const DecodeArgs p) {
  constexpr int STAGES = DPipe<NT>::STAGES, STAGE = DPipe<NT>::STAGE;
  constexpr int NBUF = DPipe<NT>::NBUF;
  constexpr int KSUB = (MODE == 1) ? 1 : 2;  // promotions per 128-wide K stage
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES], tfull[MAX_NBUF],
      tempty[MAX_NBUF], sc_full[SC_SLOTS], sc_empty[SC_SLOTS];
  __shared__ __align__(16) float sc_ring[SC_SLOTS][SC_STRIDE];
  __shared__ int s_toff[kMaxE + 1], s_off[kMaxE + 1];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;
  __shared__ float upbuf[64][DN + 1];
  __shared__ float colmax[2][DN];

  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t K = MODE == 1 ? p.H : p.I;
  const int64_t nkb = K / DK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], EPI_WARPS);
    }
    for (int s = 0; s < SC_SLOTS; ++s) {
      mbar_init(&sc_full[s], 32);  // every lane of the producer warp arrives
      mbar_init(&sc_empty[s], EPI_WARPS);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, DPipe<NT>::TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  pdl_wait();  // routing and activation terms come from earlier kernels of the stream
  pdl_trigger();
  for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
    s_toff[i] = p.tile_offsets[i];
    s_off[i] = p.offsets[i];
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int64_t n_items = (int64_t)s_toff[p.E] * p.n_blocks;
  const int64_t it_lo = n_items * blockIdx.x / gridDim.x, it_hi = n_items * (blockIdx.x + 1) / gridDim.x;
  const int64_t wblocks = MODE == 1 ? 2 * p.I / 128 : p.H / 128;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA + scales
    // The whole warp walks the stages: lane 0 issues the TMA loads, every
    // lane copies (at most) one activation scale and lanes 16/17 or 0 the
    // weight scales; each lane then arrives on the slot's barrier.
    if (lane == 0) {
      for (int t = 0; t < NT; ++t) prefetch_tmap(&tm.a[t]);
      prefetch_tmap(&tm.b);
    }
    const int a_sub = lane >> 4, a_j = lane & 15;
    int stage = 0, sslot = 0;
    uint32_t phase = 0, sphase = 0;
    bool run = true;
    for (int64_t item = it_lo; item < it_hi && run; ++item) {
      const DItem c = ditem(s_toff, s_off, p.E, p.n_blocks, item);
      int64_t r0, r1, wb;
      if (MODE == 1) {
        r0 = (int64_t)c.e * 2 * p.I + (int64_t)c.nb * 64;
        r1 = r0 + p.I;
        // lane 16: gate rows' scale block, lane 17: up rows'
        wb = (lane == 16 ? 0 : p.I) / 128 + (int64_t)c.nb * 64 / 128;
      } else {
        r0 = (int64_t)c.e * p.H + (int64_t)c.nb * 128;
        r1 = r0 + 64;
        wb = c.nb;
      }
      const float *ws = p.w_scale + (int64_t)c.e * wblocks * nkb;
      const int64_t apos = c.p0 + a_j;
      for (int64_t kb = 0; kb < nkb; ++kb) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1u, &abort_flag, DWAIT_NS)) {
          abort_flag = 1;
          set_error(p.err, DEV_ERR_TIMEOUT);
          run = false;
          break;
        }
        if (lane == 0) {
          uint8_t *st = smem + (size_t)stage * STAGE;
          mbar_arrive_expect_tx(&full_bar[stage], STAGE);
          const int32_t kx = (int32_t)(kb * DK);
          tma_load_2d(st, &tm.b, kx, (int32_t)r0, &full_bar[stage]);
          tma_load_2d(st + A_BYTES / 2, &tm.b, kx, (int32_t)r1, &full_bar[stage]);
#pragma unroll
          for (int t = 0; t < NT; ++t)
            tma_load_2d(st + A_BYTES + t * B_BYTES, &tm.a[t], kx, (int32_t)c.p0, &full_bar[stage]);
        }
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }

        if (!mbar_wait(&sc_empty[sslot], sphase ^ 1u, &abort_flag, DWAIT_NS)) {
          abort_flag = 1;
          set_error(p.err, DEV_ERR_TIMEOUT);
          run = false;
          break;
        }
        float *sc = sc_ring[sslot];
        if (a_sub < KSUB && apos < p.Pmax)
          cp_async4(sc + a_sub * DN + a_j, p.act_scale + (kb * KSUB + a_sub) * p.Pmax + apos);
        if (MODE == 1 ? (lane == 16 || lane == 17) : lane == 0)
          cp_async4(sc + 2 * DN + (MODE == 1 ? lane - 16 : 0), ws + wb * nkb + kb);
        cp_async_arrive(&sc_full[sslot]);
        if (++sslot == SC_SLOTS) { sslot = 0; sphase ^= 1u; }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr int NC = DPipe<NT>::NC;
      const uint32_t idesc = idesc_e4m3_f32(DM, NC);
      int stage = 0, buf = 0;
      uint32_t phase = 0, bphase = 0;
      for (int64_t item = it_lo; item < it_hi && !abort_flag; ++item) {
        for (int64_t kb = 0; kb < nkb && !abort_flag; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, &abort_flag, DWAIT_NS)) {
            abort_flag = 1;
            set_error(p.err, DEV_ERR_TIMEOUT);
            break;
          }
          const uint32_t a = smem_u32(smem + (size_t)stage * STAGE);
          const uint32_t b = a + A_BYTES;
#pragma unroll
          for (int sub = 0; sub < KSUB; ++sub) {
            if (!mbar_wait(&tempty[buf], bphase ^ 1u, &abort_flag, DWAIT_NS)) {
              abort_flag = 1;
              set_error(p.err, DEV_ERR_TIMEOUT);
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(buf * DPipe<NT>::BUF_COLS);
#pragma unroll
            for (int kk = sub * (4 / KSUB); kk < (sub + 1) * (4 / KSUB); ++kk)
              mma_f8f6f4(d, sw128_kmajor_desc(a + kk * 32), sw128_kmajor_desc(b + kk * 32), idesc,
                         kk > sub * (4 / KSUB) ? 1u : 0u);
            mma_commit(&tfull[buf]);
            if (++buf == NBUF) { buf = 0; bphase ^= 1u; }
          }
          mma_commit(&empty_bar[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- promotion + epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // weight row of this thread within the item
    const int w_idx = 2 * DN + ((MODE == 1 && r >= 64) ? 1 : 0);
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    int buf = 0, sslot = 0;
    uint32_t bphase = 0, sphase = 0;
    bool ok = true;
    for (int64_t item = it_lo; item < it_hi; ++item) {
      const DItem c = ditem(s_toff, s_off, p.E, p.n_blocks, item);
      float acc[DN];
#pragma unroll
      for (int j = 0; j < DN; ++j) acc[j] = 0.f;
      for (int64_t kb = 0; kb < nkb && ok; ++kb) {
        if (!mbar_wait(&sc_full[sslot], sphase, &abort_flag, DWAIT_NS)) {
          abort_flag = 1;
          set_error(p.err, DEV_ERR_TIMEOUT);
          ok = false;
          break;
        }
        const float *sc = sc_ring[sslot];
        const float sw = sc[w_idx];
#pragma unroll
        for (int sub = 0; sub < KSUB; ++sub) {
          if (!mbar_wait(&tfull[buf], bphase, &abort_flag, DWAIT_NS)) {
            abort_flag = 1;
            set_error(p.err, DEV_ERR_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t v[NT * DN];
          const uint32_t ta = t_lane + (uint32_t)(buf * DPipe<NT>::BUF_COLS);
          tmem_ld_x16(ta, v);
          tmem_ld_x16(ta + DN, v + DN);
          if (NT == 3) tmem_ld_x16(ta + 2 * DN, v + 2 * DN);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[buf]);
          if (++buf == NBUF) { buf = 0; bphase ^= 1u; }
          const float4 *sa4 = reinterpret_cast<const float4 *>(sc + sub * DN);
#pragma unroll
          for (int j4 = 0; j4 < DN / 4; ++j4) {
            const float4 sa = sa4[j4];
            const float sj[4] = {sa.x, sa.y, sa.z, sa.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int j = j4 * 4 + u;
              float t = __uint_as_float(v[j]) + __uint_as_float(v[DN + j]);
              if (NT == 3) t += __uint_as_float(v[2 * DN + j]);
              acc[j] = fmaf(t, sj[u] * sw, acc[j]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sc_empty[sslot]);
        if (++sslot == SC_SLOTS) { sslot = 0; sphase ^= 1u; }
      }
      // all four epilogue warps agree before the shared buffers are touched
      ok = named_bar_and(1, 32 * EPI_WARPS, ok);
      if (!ok) break;
      const int nvalid = (int)((c.p_end - c.p0) < DN ? (c.p_end - c.p0) : DN);
      if (MODE == 1) {
        // up rows hand their sums to the gate rows of the same h outputs
        if (r >= 64)
#pragma unroll
          for (int j = 0; j < DN; ++j) upbuf[r - 64][j] = acc[j];
        named_bar_sync(1, 32 * EPI_WARPS);
        float hv[DN];
        if (r < 64) {
#pragma unroll
          for (int j = 0; j < DN; ++j) {
            if (j < nvalid) {  // the same for the whole CTA
              hv[j] = swiglu(acc[j], upbuf[r][j]);
              const float m = warp_max(fabsf(hv[j]));
              if (lane == 0) colmax[r >> 5][j] = m;
            }
          }
        }
        named_bar_sync(1, 32 * EPI_WARPS);
        if (r < 64) {
          const int64_t col = (int64_t)c.nb * 64 + r;
#pragma unroll
          for (int j = 0; j < DN; ++j) {
            if (j >= nvalid) break;
            const int ex = e4m3_block_exponent(fmaxf(colmax[0][j], colmax[1][j]));
            uint32_t cd[3];
            e4m3_terms<3>(ldexpf(hv[j], -ex), 0.f, cd);
            const int64_t pos = c.p0 + j;
            p.h_t0[pos * p.I + col] = (uint8_t)(cd[0] & 0xffu);
            p.h_t1[pos * p.I + col] = (uint8_t)(cd[1] & 0xffu);
            p.h_t2[pos * p.I + col] = (uint8_t)(cd[2] & 0xffu);
            if (r == 0) p.h_scale[(int64_t)c.nb * p.Pmax + pos] = ldexpf(1.f, ex);
          }
        }
        // upbuf / colmax are reused only after the next item's agreement barrier
      } else {
#pragma unroll
        for (int j = 0; j < DN; ++j) {
          if (j >= nvalid) break;
          p.y[(c.p0 + j) * p.H + (int64_t)c.nb * 128 + r] = acc[j];
        }
      }
    }
  }

  __syncthreads();
  if (abort_flag) {
    // let copies and MMAs still in flight land before the CTA's memory goes away
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 50000ull) {
    }
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, DPipe<NT>::TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_decode_mma(int mode, const TmapSet &tm, const int32_t *offsets,
                              const int32_t *tile_offsets, const float *act_scale,
                              const float *w_scale, int E, int64_t H, int64_t I, int64_t Pmax,
                              uint8_t *const h_terms[3], float *h_scale, float *y, int *err,
                              int64_t max_items, int sms, cudaStream_t s) {
  DecodeArgs p;
  p.offsets = offsets;
  p.tile_offsets = tile_offsets;
  p.act_scale = act_scale;
  p.w_scale = w_scale;
  p.E = E;
  p.H = H;
  p.I = I;
  p.Pmax = Pmax;
  p.n_blocks = mode == 1 ? (int)(I / 64) : (int)(H / 128);
  p.h_t0 = h_terms ? h_terms[0] : nullptr;
  p.h_t1 = h_terms ? h_terms[1] : nullptr;
  p.h_t2 = h_terms ? h_terms[2] : nullptr;
  p.h_scale = h_scale;
  p.y = y;
  p.err = err;
  const int64_t grid = max_items < sms ? max_items : sms;
  if (grid <= 0) return cudaSuccess;
  cudaError_t e;
  if (mode == 1) {
    auto k = decode_mma_kernel<1, 2>;
    if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DPipe<2>::SMEM)) != cudaSuccess) return e;
    return launch_pdl(k, dim3((unsigned)grid), dim3(DTHREADS), DPipe<2>::SMEM, s, tm, p);
  }
  auto k = decode_mma_kernel<2, 3>;
  if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DPipe<3>::SMEM)) != cudaSuccess) return e;
  return launch_pdl(k, dim3((unsigned)grid), dim3(DTHREADS), DPipe<3>::SMEM, s, tm, p);
}

}  // namespace fp8moe
