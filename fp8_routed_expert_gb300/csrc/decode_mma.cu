// Routed-expert FFN for small batches on the 5th-generation tensor cores, in
// ONE persistent launch: gate/up + SwiGLU for every (expert tile, 128 h
// outputs), then down for every (expert tile, 256 output rows).
//
// The time of a decode step goes to moving expert weight bytes (DeepSeek-
// V4.1-Flash post, "Bytes per token decide everything"), so the kernel is
// built to stream them: each item's 256 weight rows are the MMA's N = 256
// operand, loaded by TMA in 32 KiB stages and multiplied in shared memory by
// tcgen05.mma without any per-byte instruction on the SM.
//
// Operands.  B = e4m3 weight rows (one f32 scale per 128 x 128 block).
// A = the tile's activations (up to 16 positions) as e4m3 terms that share
// one power-of-two scale per (row, 128-column block):
//   gate/up: x in two terms (exact for bf16), token-major, gathered four rows
//     at a time by TMA (tile::gather4) into the first four rows of 8-row
//     128-byte-swizzle atoms: term t, position j is row 8 (j / 4) + j % 4 of
//     a 4 KiB block at 4 KiB t.  The terms are summed by the MMA itself: two
//     passes of M64 x N256 x K32 MMAs (one per term) accumulate into the same
//     rows, so the result needs no further reduction (the tensor pipe has
//     room for it: 8 MMAs of 128 cycles per 32 KiB stage).
//   down: h in three terms (about 12 bits), stacked along M so that one pass
//     covers them all: term t, position j is A row 16 t + j.  The terms' rows
//     are written to three planes of y and added by the combine kernel.
// Every 128-wide K block is accumulated in one of two TMEM buffers and
// promoted in f32 registers as partial * s_w[row block, kb] * s_act[row, kb]
// (dragon.c §8 "Round 3": the block scale is folded out of the inner
// product) while the MMA fills the other buffer.
//
// Work queue.  The items form one list: every gate/up item (tile-major), then
// every down item (tile-major).  CTAs take items from a global counter, one
// at a time, so that a CTA that finishes early takes more and the tail is at
// most one item long.  Every item, a CTA's first included, comes from the
// counter, so an item belongs only to a CTA that is already running (a CTA
// that is not yet resident holds none).  The weight producer takes the next item
// when it issues the last load of the current one and hands its index to the
// other roles through a small ring in shared memory.
// A down item needs h of its tile, i.e. every gate/up item of the tile
// (possibly other CTAs'): each gate/up item is published on a per-tile counter
// when its h is stored, and the activation producer and the epilogue of a
// down item wait (bounded) until the tile's counter is complete.  Every
// gate/up item precedes every down item in the list and an item is taken only
// by a running CTA, which finishes it without waiting on later items, so the
// waits end.
//
// Accumulator layout (M = 64, one CTA): row 16 q + l sits in TMEM lane
// 32 q + l for l < 16.  The epilogue reads it with tcgen05.ld.16x64b: in the
// warp of lane quarter q, thread t holds row 16 q + (t >> 2) + 8 (t & 1) and,
// of every 64 columns, those with parity (t >> 1) & 1, so the two threads of
// a row (t and t ^ 2) split its columns.
// Warps: 0 weight TMA and item queue; 1 TMEM allocation and MMA issue;
// 2 activation TMA; 4..11 promotion (warp w reads lane quarter w % 4 and
// column half (w - 4) / 4): quarters 0, 1 for gate/up, 0..2 for down.  The
// gate/up tail (SwiGLU, h quantisation, stores, publication) runs on warps 7
// and 11, fed through a shared-memory hand-off, so the promoting warps start
// the next item at once and the MMA never waits for a tail; 3 idle.  The
// producer and MMA loops are warp-uniform (lane 0 issues).  Every mbarrier
// wait and counter wait is bounded by wall-clock time, and the epilogue warps
// synchronise only through mbarriers, so a wait that gives up cannot leave
// another warp stuck at a barrier.
#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace fp8moe {
using namespace sm100;

namespace {

constexpr int BM = 64;                 // MMA M: stacked activation rows
constexpr int TP = kDecodeTileN;       // positions per tile (16)
constexpr int BN = 256;                // weight rows per item
constexpr int BK = 128;                // K per stage
constexpr int A_BYTES = BM * BK;       // 8 KiB
constexpr int B_BYTES = BN * BK;       // 32 KiB
constexpr int STAGE = A_BYTES + B_BYTES;
constexpr int STAGES = 5;
constexpr uint32_t TMEM_COLS = 512;    // two 256-column accumulators
constexpr int EPI_WARPS = 8;
constexpr int HB_LD = 256 + 4;         // gate/up hand-off rows (padded against bank conflicts)
constexpr int HB_FLOATS = TP * HB_LD;  // 16.3 KiB
constexpr int kTailWarps = 2;          // warps 7 and 11
constexpr uint32_t kTemptyArrivals = 6;
constexpr int kMaxE = 1024;
constexpr int DTHREADS = 32 * 12;
constexpr size_t DSMEM = (size_t)STAGES * STAGE + HB_FLOATS * 4 + 1024;
constexpr uint64_t DWAIT_NS = 2000000000ull;

static_assert(TP == 16, "tiles of 16 positions: 4 gather atoms per x term, 16 rows per h term");

struct FfnArgs {
  const int32_t *offsets, *tile_offsets;  // tile offsets in units of TP-position tiles
  const int32_t *perm;                    // position -> pair id t * k + r
  int k;
  const float *x_scale;                   // [H/128][x_ld] per token
  int64_t x_ld;
  const float *s13, *s2;
  int E;
  int64_t H, I, Pmax;
  uint8_t *h_t0, *h_t1, *h_t2;            // [Pmax, I] three terms of h
  float *h_scale;                         // [I/128][Pmax]
  float *y;                               // three term planes [3][y_plane]: [P, H] each
  int64_t y_plane;
  int32_t *done13;                        // finished gate/up items per tile (0 at entry)
  int32_t *queue;                         // items handed out so far (0 at entry)
  int *err;
  const int32_t *slot_of;                 // weight slab of each expert, or nullptr (slab = expert)
};

struct DItem {
  int e, nb;
  int64_t tile;       // global tile index
  int64_t p0;         // first position of the tile
  int nvalid;         // positions of this tile (1..TP)
};

__device__ __forceinline__ DItem ditem(const int *toff, const int *off, int E, int n_blocks, int64_t item) {
  DItem c;
  c.tile = item / n_blocks;
  c.nb = (int)(item % n_blocks);
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (toff[mid] <= c.tile) lo = mid;
    else hi = mid;
  }
  c.e = lo;
  c.p0 = off[lo] + (c.tile - toff[lo]) * TP;
  const int64_t n = off[lo + 1] - c.p0;
  c.nvalid = (int)(n < TP ? n : TP);
  return c;
}

// The item list: gate/up items [0, n1), then down items [n1, n).
struct Work {
  int64_t n1, n;
  int nb1, nb2;  // column blocks per tile: I/128 (gate/up), H/256 (down)
  __device__ __forceinline__ bool down(int64_t i) const { return i >= n1; }
  __device__ __forceinline__ int64_t local(int64_t i) const { return i < n1 ? i : i - n1; }
  __device__ __forceinline__ int nblocks(int64_t i) const { return i < n1 ? nb1 : nb2; }
};

constexpr int QD = 4;  // item ring depth

// Consumer side of the item ring: the whole warp waits (bounded) for slot
// `slot`, reads the item (-1: end of the list) and lane 0 releases the slot.
// Returns false when the wait gave up.
__device__ __forceinline__ bool take_item(const volatile int64_t *s_item, uint64_t *full, uint64_t *empty,
                                          int &slot, uint32_t &qphase, volatile int *abort_flag,
                                          int64_t *item) {
  if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], qphase, abort_flag, DWAIT_NS))) return false;
  *item = s_item[slot];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&empty[slot]);
  if (++slot == QD) {
    slot = 0;
    qphase ^= 1u;
  }
  return true;
}

// Four rows of a 2-D tensor (box of one row) into consecutive 128-byte rows
// of shared memory; the destination is the start of a 1024-byte swizzle atom.
__device__ __forceinline__ void tma_gather4(void *dst, const CUtensorMap *m, int32_t x, int32_t r0,
                                            int32_t r1, int32_t r2, int32_t r3, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
      "r"(smem_u32(bar))
      : "memory");
}

// Butterfly exchange with lane ^ 2, and a 16-byte global store, both as
// volatile asm so that they stay in program order.
__device__ __forceinline__ float shfl_xor2_ordered(float v) {
  float r;
  asm volatile("shfl.sync.bfly.b32 %0, %1, 2, 0x1f, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ void st_global_f4_ordered(float *p, float4 v) {
  asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

__device__ __forceinline__ void fail(volatile int *abort_flag, int *err) {
  *abort_flag = 1;
  set_error(err, DEV_ERR_TIMEOUT);
}

// Lane 0 waits (bounded) until the tile's gate/up items are all published;
// the outcome is broadcast to the warp.
__device__ __forceinline__ bool wait_tile(const int32_t *done13, int64_t tile, int need,
                                          volatile int *abort_flag) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) {
    ok = wait_counter_ge(done13 + tile, need, abort_flag, DWAIT_NS);
    fence_proxy_async_global();
  }
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// 16 lanes x 64 columns (tcgen05.ld.16x64b.x32, no wait): value i of thread
// t is lane (t >> 2) + 8 (t & 1), column 2 i + ((t >> 1) & 1).
__device__ __forceinline__ void tmem_ld16x64(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x64b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(DTHREADS, 1) decode_ffn_kernel(const __grid_constant__ DecodeMaps tm,
                                                                 const FfnArgs p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_a[STAGES], full_b[STAGES], empty_bar[STAGES], tfull[2], tempty[2];
  __shared__ __align__(8) uint64_t item_full[QD], item_empty[QD], hfull, hempty;
  __shared__ volatile int64_t s_item[QD];
  __shared__ int s_toff[kMaxE + 1], s_off[kMaxE + 1];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;
  __shared__ int32_t s_rows[TP];   // token rows of the activation producer's current tile

  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float *hbuf = reinterpret_cast<float *>(smem + (size_t)STAGES * STAGE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nkb1 = p.H / BK, nkb2 = p.I / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_a[s], 1);
      mbar_init(&full_b[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kTemptyArrivals);
    }
    mbar_init(&hfull, 4);            // gate/up promoters
    mbar_init(&hempty, kTailWarps);  // tail warps
    for (int b = 0; b < QD; ++b) {
      mbar_init(&item_full[b], 1);
      mbar_init(&item_empty[b], 2 + EPI_WARPS);  // activation producer, MMA, epilogue warps
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  pdl_wait();  // routing and activation terms come from the previous kernel
  pdl_trigger();
  for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
    s_toff[i] = p.tile_offsets[i];
    s_off[i] = p.offsets[i];
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  Work wk;
  wk.nb1 = (int)(p.I / 128);
  wk.nb2 = (int)(p.H / 256);
  wk.n1 = (int64_t)s_toff[p.E] * wk.nb1;
  wk.n = wk.n1 + (int64_t)s_toff[p.E] * wk.nb2;

  if (warp == 0) {
    // ---------------------------------------------------------------- weight TMA + item queue
    if (lane == 0) {
      prefetch_tmap(&tm.w13);
      prefetch_tmap(&tm.w2);
    }
    int stage = 0, slot = 0;
    uint32_t phase = 0, qphase = 0;
    int64_t item = 0;  // every item comes from the queue, the first one included
    if (lane == 0) item = atomicAdd(p.queue, 1);
    item = __shfl_sync(0xffffffffu, item, 0);
    bool run = true;
    while (run) {
      // hand the item to the other roles
      if (!__all_sync(0xffffffffu, mbar_wait(&item_empty[slot], qphase ^ 1u, &abort_flag, DWAIT_NS))) {
        if (lane == 0) fail(&abort_flag, p.err);
        break;
      }
      const bool end = item >= wk.n;
      if (lane == 0) {
        s_item[slot] = end ? -1 : item;
        mbar_arrive(&item_full[slot]);
      }
      __syncwarp();
      if (++slot == QD) {
        slot = 0;
        qphase ^= 1u;
      }
      if (end) break;
      const bool dn = wk.down(item);
      const DItem c = ditem(s_toff, s_off, p.E, wk.nblocks(item), wk.local(item));
      const int64_t ws = p.slot_of ? __ldg(p.slot_of + c.e) : c.e;      // weight slab
      const int64_t r0 = dn ? ws * p.H + (int64_t)c.nb * 256         // 256 W2 rows
                            : ws * 2 * p.I + (int64_t)c.nb * 128;    // 128 gate rows
      const int64_t nkb = dn ? nkb2 : nkb1;
      int next = 0;
      for (int64_t kb = 0; kb < nkb; ++kb) {
        if (!__all_sync(0xffffffffu, mbar_wait(&empty_bar[stage], phase ^ 1u, &abort_flag, DWAIT_NS))) {
          if (lane == 0) fail(&abort_flag, p.err);
          run = false;
          break;
        }
        if (lane == 0) {
          // the next item is taken with the last load of this one
          if (kb == nkb - 1) next = atomicAdd(p.queue, 1);
          uint8_t *sb = smem + (size_t)stage * STAGE + A_BYTES;
          mbar_arrive_expect_tx(&full_b[stage], B_BYTES);
          const int32_t kx = (int32_t)(kb * BK);
          if (dn) {
            tma_load_2d(sb, &tm.w2, kx, (int32_t)r0, &full_b[stage]);
          } else {
            tma_load_2d(sb, &tm.w13, kx, (int32_t)r0, &full_b[stage]);                      // gate
            tma_load_2d(sb + B_BYTES / 2, &tm.w13, kx, (int32_t)(r0 + p.I), &full_b[stage]);  // up
          }
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      item = __shfl_sync(0xffffffffu, next, 0);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- activation TMA
    if (lane == 0) {
      prefetch_tmap(&tm.x[0]);
      prefetch_tmap(&tm.x[1]);
      for (int t = 0; t < 3; ++t) prefetch_tmap(&tm.h[t]);
    }
    int stage = 0, slot = 0;
    uint32_t phase = 0, qphase = 0;
    bool run = true;
    while (run) {
      int64_t item;
      if (!take_item(s_item, item_full, item_empty, slot, qphase, &abort_flag, &item)) {
        if (lane == 0) fail(&abort_flag, p.err);
        break;
      }
      if (item < 0) break;
      const bool dn = wk.down(item);
      const DItem c = ditem(s_toff, s_off, p.E, wk.nblocks(item), wk.local(item));
      const int64_t nkb = dn ? nkb2 : nkb1;
      if (!dn) {
        // token of each of the tile's positions; padding positions repeat
        // the tile's first token and their rows are never read back
        __syncwarp();
        if (lane < TP) s_rows[lane] = __ldg(p.perm + c.p0 + (lane < c.nvalid ? lane : 0)) / p.k;
        __syncwarp();
      } else if (!wait_tile(p.done13, c.tile, kTailWarps * wk.nb1, &abort_flag)) {
        if (lane == 0) fail(&abort_flag, p.err);
        break;
      }
      const int n_atoms = (c.nvalid + 3) / 4;
      for (int64_t kb = 0; kb < nkb; ++kb) {
        if (!__all_sync(0xffffffffu, mbar_wait(&empty_bar[stage], phase ^ 1u, &abort_flag, DWAIT_NS))) {
          if (lane == 0) fail(&abort_flag, p.err);
          run = false;
          break;
        }
        if (lane == 0) {
          uint8_t *sa = smem + (size_t)stage * STAGE;
          const int32_t kx = (int32_t)(kb * BK);
          if (!dn) {
            mbar_arrive_expect_tx(&full_a[stage], (uint32_t)(2 * n_atoms * 512));
            for (int t = 0; t < 2; ++t)
              for (int g = 0; g < n_atoms; ++g)  // atom 4 t + g: 1024-byte aligned
                tma_gather4(sa + (4 * t + g) * 1024, &tm.x[t], kx, s_rows[4 * g], s_rows[4 * g + 1],
                            s_rows[4 * g + 2], s_rows[4 * g + 3], &full_a[stage]);
          } else {
            mbar_arrive_expect_tx(&full_a[stage], 3 * TP * BK);
#pragma unroll
            for (int t = 0; t < 3; ++t)
              tma_load_2d(sa + t * TP * BK, &tm.h[t], kx, (int32_t)c.p0, &full_a[stage]);
          }
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    const uint32_t idesc = idesc_e4m3_f32(BM, BN);
    int stage = 0, buf = 0, slot = 0;
    uint32_t phase = 0, bphase = 0, qphase = 0;
    bool run = true;
    while (run) {
      int64_t item;
      if (!take_item(s_item, item_full, item_empty, slot, qphase, &abort_flag, &item)) {
        if (lane == 0) fail(&abort_flag, p.err);
        break;
      }
      if (item < 0) break;
      const bool dn = wk.down(item);
      const int64_t nkb = dn ? nkb2 : nkb1;
      for (int64_t kb = 0; kb < nkb; ++kb) {
        const bool ready = mbar_wait(&full_b[stage], phase, &abort_flag, DWAIT_NS) &&
                           mbar_wait(&full_a[stage], phase, &abort_flag, DWAIT_NS) &&
                           mbar_wait(&tempty[buf], bphase ^ 1u, &abort_flag, DWAIT_NS);
        if (!__all_sync(0xffffffffu, ready)) {
          if (lane == 0) fail(&abort_flag, p.err);
          run = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a = smem_u32(smem + (size_t)stage * STAGE);
          const uint64_t bdesc = sw128_kmajor_desc(a + A_BYTES);
          const uint32_t d = tmem + (uint32_t)(buf * BN);
          // down: one pass over the M-stacked h terms; gate/up: one pass per x
          // term (4 KiB apart), accumulating into the same rows.  A term's
          // M = 64 operand runs past its 32 rows into the next term / the B
          // tile: those output rows are never read.
          const int n_pass = dn ? 1 : 2;
          for (int t = 0; t < n_pass; ++t) {
            const uint64_t adesc = sw128_kmajor_desc(a + (uint32_t)t * 4096u);
#pragma unroll
            for (int kk = 0; kk < BK / 32; ++kk)  // the descriptors' address field counts 16 bytes
              mma_f8f6f4(d, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc,
                         (t > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&empty_bar[stage]);
          mma_commit(&tfull[buf]);
        }
        __syncwarp();
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        buf ^= 1;
        if (buf == 0) bphase ^= 1u;
      }
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- promotion + epilogue
    const int quarter = warp & 3;      // TMEM lanes 32 quarter .. + 15
    const int half = (warp - 4) >> 2;  // column half of the 256-wide item
    const int rq = (lane >> 2) + 8 * (lane & 1);  // row within the quarter
    const int par = (lane >> 1) & 1;   // parity of this thread's columns
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    int slot = 0;
    uint32_t qphase = 0, hphase = 0;
    uint64_t kbc = 0;  // K blocks of all items so far: TMEM buffer kbc & 1, phase (kbc >> 1) & 1
    while (true) {
      int64_t item;
      if (!take_item(s_item, item_full, item_empty, slot, qphase, &abort_flag, &item)) {
        if (lane == 0) fail(&abort_flag, p.err);
        break;
      }
      if (item < 0) break;
      const bool dn = wk.down(item);
      const DItem c = ditem(s_toff, s_off, p.E, wk.nblocks(item), wk.local(item));
      const int64_t nkb = dn ? nkb2 : nkb1;
      // Warps of quarters 0..2 follow every K block of every item (their
      // waits on the TMEM buffers stay in phase order, and each block gets
      // exactly 6 arrivals); they promote the rows they hold: quarters 0, 1
      // for gate/up (both x terms summed by the MMA), 0..2 for down (term =
      // quarter).  Quarter 3 never touches the TMEM buffers.
      if (quarter == 3) {
        if (!dn) {
          // ------------------------------------------------ gate/up tail:
          // h = silu(gate) * up, three e4m3 terms with one power-of-two scale
          // per (position, 128 outputs), stores, publication.  Thread tau of
          // warps 7 and 11: position tau / 4, outputs 32 (tau % 4) .. + 31.
          const bool got = __all_sync(0xffffffffu, mbar_wait(&hfull, hphase, &abort_flag, DWAIT_NS));
          if (!got && lane == 0) fail(&abort_flag, p.err);
          const int tau = (warp == 11 ? 32 : 0) + lane;
          const int j = tau >> 2, sg = tau & 3;
          float hv[32];
          {
            const float *gr = hbuf + j * HB_LD + 32 * sg;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float4 g4 = *reinterpret_cast<const float4 *>(gr + i);
              const float4 u4 = *reinterpret_cast<const float4 *>(gr + 128 + i);
              hv[i] = swiglu(g4.x, u4.x);
              hv[i + 1] = swiglu(g4.y, u4.y);
              hv[i + 2] = swiglu(g4.z, u4.z);
              hv[i + 3] = swiglu(g4.w, u4.w);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&hempty);
          hphase ^= 1u;
          const bool valid = got && j < c.nvalid;
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(hv[i]));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
          if (valid) {
            const int ex = e4m3_block_exponent(amax);
            const Pow2 down = pow2_factors(-ex);
            const int64_t pos = c.p0 + j;
            const int64_t off = pos * p.I + (int64_t)c.nb * 128 + 32 * sg;
#pragma unroll
            for (int g = 0; g < 2; ++g) {  // 16 outputs: one 16-byte store per term
              uint32_t w[3][8];
#pragma unroll
              for (int m = 0; m < 8; ++m) {
                uint32_t t3[3];
                e4m3_terms<3>(down(hv[16 * g + 2 * m]), down(hv[16 * g + 2 * m + 1]), t3);
#pragma unroll
                for (int t = 0; t < 3; ++t) w[t][m] = t3[t];
              }
#pragma unroll
              for (int t = 0; t < 3; ++t) {
                uint8_t *dst = (t == 0 ? p.h_t0 : (t == 1 ? p.h_t1 : p.h_t2)) + off + 16 * g;
                *reinterpret_cast<uint4 *>(dst) = make_uint4(w[t][0] | (w[t][1] << 16), w[t][2] | (w[t][3] << 16),
                                                             w[t][4] | (w[t][5] << 16), w[t][6] | (w[t][7] << 16));
              }
            }
            if (sg == 0) p.h_scale[(int64_t)c.nb * p.Pmax + pos] = ldexpf(1.f, ex);
          }
          // publish this warp's half of the item: every lane orders its h
          // stores before later async-proxy (TMA) reads, then lane 0's
          // gpu-scope fence (cumulative over the warp) and counter increment
          fence_proxy_async_global();
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            atomicAdd(p.done13 + c.tile, 1);
          }
        }
        continue;
      }
      // this thread's row: position j (gate/up: rows 4..7 of each gather
      // atom are never filled, so only lanes < 16 hold positions) or
      // position rq of term quarter (down)
      const int j = dn ? rq : 8 * (quarter & 1) + 4 * (lane & 1) + (lane >> 2);
      const bool valid = (dn || (quarter < 2 && lane < 16)) && j < c.nvalid;
      const int64_t pos = c.p0 + (valid ? j : 0);
      const float *sa_p;
      int64_t sa_ld;
      if (!dn) {
        sa_p = p.x_scale + __ldg(p.perm + pos) / p.k;
        sa_ld = p.x_ld;
      } else {
        // h and its scales are written in this launch by other CTAs: acquire
        // the tile's counter before reading them, and read them coherently
        if (!wait_tile(p.done13, c.tile, kTailWarps * wk.nb1, &abort_flag)) fail(&abort_flag, p.err);
        sa_p = p.h_scale + pos;
        sa_ld = p.Pmax;
      }
      // weight scale rows of this half's two 64-column chunks: gate / up
      // rows (gate/up) or the half's 128-row block (down)
      const float *wsc = dn ? p.s2 + (int64_t)c.e * (p.H / 128) * nkb2
                            : p.s13 + (int64_t)c.e * (2 * p.I / 128) * nkb1;
      const int64_t wb0 = dn ? 2 * (int64_t)c.nb + half : c.nb;
      const int64_t wb1 = dn ? 2 * (int64_t)c.nb + half : p.I / 128 + c.nb;
      // columns of this half's two chunks
      const uint32_t col0 = dn ? 128u * half : 64u * half;
      const uint32_t col1 = dn ? 128u * half + 64u : 128u + 64u * half;
      auto ld_sa = [&](int64_t kb) -> float {
        return dn ? __ldcg(sa_p + kb * sa_ld) : __ldg(sa_p + kb * sa_ld);
      };
      const bool rows = dn || quarter < 2;  // this warp's TMEM rows hold results
      // acc[i] = column col0 + 2 i + par, acc[32 + i] = column col1 + 2 i + par
      float acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = 0.f;
      float sa_n = ld_sa(0), s0_n = __ldg(wsc + wb0 * nkb), s1_n = __ldg(wsc + wb1 * nkb);
      bool ok = true;
      for (int64_t kb = 0; kb < nkb; ++kb) {
        const float sa = sa_n, c0 = sa * s0_n, c1 = sa * s1_n;
        if (kb + 1 < nkb) {  // next block's scales, in flight while this one is promoted
          sa_n = ld_sa(kb + 1);
          s0_n = __ldg(wsc + wb0 * nkb + kb + 1);
          s1_n = __ldg(wsc + wb1 * nkb + kb + 1);
        }
        const int buf = (int)(kbc & 1);
        if (ok && !mbar_wait(&tfull[buf], (uint32_t)(kbc >> 1) & 1u, &abort_flag, DWAIT_NS)) {
          fail(&abort_flag, p.err);
          ok = false;
        }
        tc_fence_after();
        const uint32_t tb = t_lane + (uint32_t)(buf * BN);
        if (rows) {
          float v[32];
          tmem_ld16x64(tb + col0, v);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = fmaf(v[i], c0, acc[i]);
          tmem_ld16x64(tb + col1, v);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[32 + i] = fmaf(v[i], c1, acc[32 + i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        ++kbc;
      }
      if (!rows) continue;
      if (!dn) {
        // hand gate and up to the tail warps: hbuf[j][o] gate, [j][128 + o] up
        if (!__all_sync(0xffffffffu, mbar_wait(&hempty, hphase ^ 1u, &abort_flag, DWAIT_NS)) && lane == 0)
          fail(&abort_flag, p.err);
        if (lane < 16) {
          float *hr = hbuf + j * HB_LD;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            hr[col0 + 2 * i + par] = acc[i];
            hr[col1 + 2 * i + par] = acc[32 + i];
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&hfull);
        hphase ^= 1u;
      } else {
        // y term `quarter`: the pair (lane, lane ^ 2) holds the even / odd
        // columns of a row; each assembles four consecutive ones in turn
        float *dy = p.y + (int64_t)quarter * p.y_plane + pos * p.H + (int64_t)c.nb * 256;
        // (volatile shuffles and stores keep the compiler from hoisting all
        // 64 exchanges ahead of the stores)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const uint32_t cb = h2 ? col1 : col0;
#pragma unroll
          for (int m2 = 0; m2 < 16; m2 += 2) {
            // m = m2 is assembled by the even thread, m2 + 1 by the odd one:
            // each sends the pair the other needs
            const int i0 = 32 * h2 + 2 * m2;  // pair m2 at i0, i0 + 1; pair m2 + 1 at i0 + 2, i0 + 3
            const float mine0 = par ? acc[i0 + 2] : acc[i0], mine1 = par ? acc[i0 + 3] : acc[i0 + 1];
            const float oth0 = par ? acc[i0] : acc[i0 + 2], oth1 = par ? acc[i0 + 1] : acc[i0 + 3];
            const float o0 = shfl_xor2_ordered(oth0), o1 = shfl_xor2_ordered(oth1);
            const float4 v = par ? make_float4(o0, mine0, o1, mine1) : make_float4(mine0, o0, mine1, o1);
            if (valid) st_global_f4_ordered(dy + cb + 4 * (m2 + par), v);
          }
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
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_decode_ffn(const DecodeMaps &maps, const int32_t *offsets,
                              const int32_t *tile_offsets, const int32_t *perm, int k,
                              const float *x_scale, int64_t x_ld, const float *s13, const float *s2,
                              int E, int64_t H, int64_t I, int64_t Pmax, uint8_t *const h_terms[3],
                              float *h_scale, float *y, int64_t y_plane, int32_t *done13, int *err,
                              int64_t max_tiles, int sms, cudaStream_t s, const int32_t *slot_of) {
  FfnArgs p;
  p.slot_of = slot_of;
  p.offsets = offsets;
  p.tile_offsets = tile_offsets;
  p.perm = perm;
  p.k = k;
  p.x_scale = x_scale;
  p.x_ld = x_ld;
  p.s13 = s13;
  p.s2 = s2;
  p.E = E;
  p.H = H;
  p.I = I;
  p.Pmax = Pmax;
  p.h_t0 = h_terms[0];
  p.h_t1 = h_terms[1];
  p.h_t2 = h_terms[2];
  p.h_scale = h_scale;
  p.y = y;
  p.y_plane = y_plane;
  p.done13 = done13;
  p.queue = done13 + max_tiles;
  p.err = err;
  if (E > kMaxE || H % 256 != 0) return cudaErrorInvalidValue;
  const int64_t max_items = max_tiles * (H / 256 > I / 128 ? H / 256 : I / 128);
  const int64_t grid = max_items < sms ? max_items : sms;
  if (grid <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(decode_ffn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DSMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_ffn_kernel, dim3((unsigned)grid), dim3(DTHREADS), DSMEM, s, maps, p);
}

}  // namespace fp8moe
