// Router logits of large batches on the 5th-generation tensor cores.
//
// logits[t, e] = sum_h x[t, h] W[e, h] with x bf16 and W f32 (dragon.c,
// "Precision": router f32).  W is split exactly into three bf16 terms,
// W = W0 + W1 + W2 (W0 = bf16(W), W1 = bf16(W - W0), W2 = W - W0 - W1, which
// has at most 8 significant bits), so that every product x * Wi is exact in
// f32, and the three terms are summed by tcgen05.mma kind::f16 (bf16 x bf16,
// f32 accumulate) into one TMEM accumulator.  To keep the rounding chain of
// every logit short -- its length enters the error bound that certifies the
// top-k selection (the exact path takes the tokens it cannot certify) --
// each 128-wide K block is accumulated in its own TMEM buffer (24 MMA
// instructions) and added to f32 registers by the epilogue, K blocks in
// ascending order; a K range split over CTAs lands in separate planes that
// the selection adds in plane order.
//
// Tile: 128 tokens x 128 experts, K staged 64 at a time (one 128-byte row
// of bf16: 16 KiB of x and 3 x 16 KiB of W terms per stage, three stages);
// four 128-column TMEM buffers let the MMA run three K blocks ahead.  Warp
// 0 issues TMA, warp 1 allocates TMEM and issues the MMAs, warps 2..9 add
// the K blocks and store the logits.  Every wait is bounded.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace fp8moe {
using namespace sm100;

namespace {

constexpr int RBM = 128, RBN = 128, RBK = 64;  // tokens, experts, K per stage
constexpr int R_TERMS = 3;
constexpr int R_A = RBM * RBK * 2;              // 16 KiB of x
constexpr int R_B = RBN * RBK * 2;              // 16 KiB per W term
constexpr int R_STAGE = R_A + R_TERMS * R_B;    // 64 KiB
constexpr int R_STAGES = 3;
constexpr int R_EPI = 8;
constexpr int R_THREADS = 64 + 32 * R_EPI;
constexpr int R_BUFS = 4;                       // TMEM buffers of 128 columns
constexpr uint32_t R_TMEM = 512;
constexpr size_t R_SMEM = (size_t)R_STAGES * R_STAGE + 1024;
constexpr uint64_t R_WAIT_NS = 2000000000ull;
// MMA instructions per 128-wide K block: 2 stages x 4 K steps of 16 x 3 terms
constexpr int R_MMAS_PER_KB = 2 * (RBK / 16) * R_TERMS;

// Instruction descriptor of kind::f16: D f32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct RArgs {
  int64_t T, E, H;
  int ks;            // planes of the K split
  int n_tt, n_et;    // token and expert tiles
  int64_t n_items;   // ks * n_tt * n_et
  float *logits;     // [ks][T][E]
  int *err;
};

struct RItem {
  int z, tt, et;
  int64_t kb_lo, kb_hi;  // 128-wide K blocks of this plane
};

__device__ __forceinline__ RItem ritem(const RArgs &p, int64_t item) {
  RItem r;
  r.et = (int)(item % p.n_et);
  r.tt = (int)((item / p.n_et) % p.n_tt);
  r.z = (int)(item / ((int64_t)p.n_et * p.n_tt));
  const int64_t nkb = p.H / 128;
  r.kb_lo = nkb * r.z / p.ks;
  r.kb_hi = nkb * (r.z + 1) / p.ks;
  return r;
}

__global__ void __launch_bounds__(R_THREADS, 1) router_tc_kernel(const __grid_constant__ CUtensorMap tx,
                                                                 const __grid_constant__ CUtensorMap tw,
                                                                 const RArgs p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[R_STAGES], empty_bar[R_STAGES], tfull[R_BUFS], tempty[R_BUFS];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < R_STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < R_BUFS; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], R_EPI);
    }
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tx);
    prefetch_tmap(&tw);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, R_TMEM);
    tmem_relinquish();
    tc_fence_before();
  }
  pdl_wait();  // the split W terms come from the previous kernel
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int64_t item = blockIdx.x; item < p.n_items && !abort_flag; item += gridDim.x) {
        const RItem r = ritem(p, item);
        for (int64_t kb = r.kb_lo; kb < r.kb_hi && !abort_flag; ++kb) {
          for (int hs = 0; hs < 2; ++hs) {
            if (!mbar_wait(&empty_bar[stage], phase ^ 1u, &abort_flag, R_WAIT_NS)) {
              abort_flag = 1;
              set_error(p.err, DEV_ERR_TIMEOUT);
              break;
            }
            uint8_t *st = smem + (size_t)stage * R_STAGE;
            mbar_arrive_expect_tx(&full_bar[stage], R_STAGE);
            const int32_t kx = (int32_t)(kb * 128 + hs * RBK);
            tma_load_2d(st, &tx, kx, r.tt * RBM, &full_bar[stage]);
#pragma unroll
            for (int t = 0; t < R_TERMS; ++t)
              tma_load_2d(st + R_A + t * R_B, &tw, kx, (int32_t)(t * p.E + (int64_t)r.et * RBN),
                          &full_bar[stage]);
            if (++stage == R_STAGES) { stage = 0; phase ^= 1u; }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(RBM, RBN);
      int stage = 0, buf = 0;
      uint32_t phase = 0, bphase = 0;
      for (int64_t item = blockIdx.x; item < p.n_items && !abort_flag; item += gridDim.x) {
        const RItem r = ritem(p, item);
        for (int64_t kb = r.kb_lo; kb < r.kb_hi && !abort_flag; ++kb) {
          if (!mbar_wait(&tempty[buf], bphase ^ 1u, &abort_flag, R_WAIT_NS)) {
            abort_flag = 1;
            set_error(p.err, DEV_ERR_TIMEOUT);
            break;
          }
          const uint32_t d = tmem + (uint32_t)buf * RBN;
          bool ok = true;
          for (int hs = 0; hs < 2; ++hs) {
            if (!mbar_wait(&full_bar[stage], phase, &abort_flag, R_WAIT_NS)) {
              abort_flag = 1;
              set_error(p.err, DEV_ERR_TIMEOUT);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(smem + (size_t)stage * R_STAGE);
#pragma unroll
            for (int kk = 0; kk < RBK / 16; ++kk) {  // 16 bf16 = 32 bytes per K step
              const uint64_t ad = sw128_kmajor_desc(a0 + kk * 32);
#pragma unroll
              for (int t = 0; t < R_TERMS; ++t)
                mma_bf16(d, ad, sw128_kmajor_desc(a0 + R_A + t * R_B + kk * 32), idesc,
                         (hs > 0 || kk > 0 || t > 0) ? 1u : 0u);
            }
            mma_commit(&empty_bar[stage]);
            if (++stage == R_STAGES) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          mma_commit(&tfull[buf]);
          if (++buf == R_BUFS) { buf = 0; bphase ^= 1u; }
        }
      }
    }
  } else {
    // warps 2..9: lane quarter warp % 4, column half (warp - 2) / 4
    const int quarter = warp & 3, chalf = (warp - 2) >> 2;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    int buf = 0;
    uint32_t bphase = 0;
    for (int64_t item = blockIdx.x; item < p.n_items; item += gridDim.x) {
      const RItem r = ritem(p, item);
      float acc[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0.f;
      bool ok = true;
      for (int64_t kb = r.kb_lo; kb < r.kb_hi; ++kb) {
        if (!mbar_wait(&tfull[buf], bphase, nullptr, R_WAIT_NS)) {
          abort_flag = 1;
          set_error(p.err, DEV_ERR_TIMEOUT);
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          float v[16];
          tmem_ld_32x32b_x16(t_lane + (uint32_t)(buf * RBN + chalf * 64 + ch * 16), v);
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[ch * 16 + j] += v[j];  // K blocks in ascending order
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        if (++buf == R_BUFS) { buf = 0; bphase ^= 1u; }
      }
      if (!ok) break;
      const int64_t t = (int64_t)r.tt * RBM + quarter * 32 + lane;
      if (t < p.T) {
        float *dst = p.logits + ((int64_t)r.z * p.T + t) * p.E;
        const int64_t e0 = (int64_t)r.et * RBN + chalf * 64;
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (e0 + j < p.E) dst[e0 + j] = acc[j];
      }
    }
  }

  __syncthreads();
  if (abort_flag) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 50000ull) {
    }
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, R_TMEM);
  }
}

// W f32 [E, H] -> three bf16 terms [3][E, H] whose sum is W exactly.
__global__ void __launch_bounds__(256) split_w_kernel(const float *__restrict__ W, int64_t n,
                                                      __nv_bfloat16 *__restrict__ terms) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float w = W[i];
    const __nv_bfloat16 t0 = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(t0);  // exact
    const __nv_bfloat16 t1 = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(t1);  // exact, at most 8 significant bits
    terms[i] = t0;
    terms[n + i] = t1;
    terms[2 * n + i] = __float2bfloat16_rn(r2);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void *q = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) ==
            cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(q);
  }
  return fn;
}

}  // namespace

// Row-major bf16 matrix [rows, cols], boxes of 128 rows x 64 columns (128
// bytes), 128-byte swizzle; rows past the end read as zero.
bool encode_bf16_tmap(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int router_tc_k_split(int64_t T, int64_t E, int64_t H, int sms) {
  const int64_t tiles = ((T + RBM - 1) / RBM) * ((E + RBN - 1) / RBN);
  int64_t ks = (sms + tiles - 1) / tiles;
  const int64_t nkb = H / 128;
  if (ks > nkb) ks = nkb;
  if (ks > kRouterMaxKSplit) ks = kRouterMaxKSplit;
  return ks < 1 ? 1 : (int)ks;
}

// gamma_d of the tensor-core logits: each MMA instruction is allowed 8 units
// of 2^-24 (four f32 ulps of its running sum), 24 of them per K block, then
// one f32 addition per K block, the plane additions and the bias.
float router_tc_gamma(int64_t H, int ks) {
  const double u = 1.0 / 16777216.0;
  const double d = 8.0 * R_MMAS_PER_KB + (double)(H / 128) + ks + 1;
  const double g = d * u / (1.0 - d * u);
  return nextafterf((float)(g * (1.0 + 1e-6)), INFINITY);
}

cudaError_t launch_router_logits_tc(const CUtensorMap &tx, const CUtensorMap &tw, const float *W,
                                    __nv_bfloat16 *w_terms, int64_t T, int64_t E, int64_t H, int ks,
                                    float *logits, int *err, int sms, cudaStream_t s) {
  const int64_t n = E * H;
  int64_t g = (n + 255) / 256;
  if (g > (int64_t)sms * 8) g = (int64_t)sms * 8;
  cudaError_t e = launch_pdl(split_w_kernel, dim3((unsigned)g), dim3(256), 0, s, W, n, w_terms);
  if (e != cudaSuccess) return e;
  RArgs p;
  p.T = T;
  p.E = E;
  p.H = H;
  p.ks = ks;
  p.n_tt = (int)((T + RBM - 1) / RBM);
  p.n_et = (int)((E + RBN - 1) / RBN);
  p.n_items = (int64_t)ks * p.n_tt * p.n_et;
  p.logits = logits;
  p.err = err;
  if ((e = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)R_SMEM)) != cudaSuccess)
    return e;
  const int64_t grid = p.n_items < sms ? p.n_items : sms;
  return launch_pdl(router_tc_kernel, dim3((unsigned)grid), dim3(R_THREADS), R_SMEM, s, tx, tw, p);
}

}  // namespace fp8moe
