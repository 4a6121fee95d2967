// Internal launchers of the layer's kernels (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace fp8moe {

// Launch with programmatic stream serialization (the kernel starts before
// its predecessor finishes and orders itself with griddepcontrol.wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// T at or below which the router uses one warp per expert row; above it, the
// tiled kernel.
constexpr int64_t kRouterWarpMaxT = 64;
// Rows of one grouped-GEMM tile (tile list granularity).
constexpr int kTileM = 128;

// Largest split of the router's K loop over CTAs (planes of partial logits).
constexpr int kRouterMaxKSplit = 8;
int router_chain_depth(int64_t H);
// gamma_d = d u / (1 - d u) of the small-batch logit kernel's longest
// rounding chain d, rounded up: the relative factor of its error bound.
float router_gamma(int64_t H);
// T <= kRouterWarpMaxT: logits, selection and the pair sort in one launch
// (ticket: an int32 that is 0 between calls).
size_t route_decode_smem(int64_t E);
cudaError_t launch_route_decode(const __nv_bfloat16 *x, int64_t T, const float *W, const float *bias,
                                int64_t E, int64_t H, int k, float gamma, float *logits, float *wnorm,
                                float *xnorm, __half *x16, float *xscale, int32_t *ticket,
                                int32_t *idx, float *wts, int32_t *counts, int32_t *offsets,
                                int32_t *perm, int32_t *inv, int32_t *active, int32_t *n_active,
                                int32_t *tile_offsets, int tile_m, uint32_t *pos_max, int *err,
                                cudaStream_t s);
// ||W_e||_2 of every router row.
cudaError_t launch_row_norms(const float *W, int64_t E, int64_t H, float *wnorm, cudaStream_t s);
// Tensor-core router logits (T > kRouterWarpMaxT): W split into three bf16
// terms (w_terms [3][E, H], whose map tw has boxes of 128 rows x 64 columns),
// x through map tx (bf16 [T, H], same boxes); ks planes [ks][T][E].
bool encode_bf16_tmap(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows);
int router_tc_k_split(int64_t T, int64_t E, int64_t H, int sms);
float router_tc_gamma(int64_t H, int ks);
cudaError_t launch_router_logits_tc(const CUtensorMap &tx, const CUtensorMap &tw, const float *W,
                                    __nv_bfloat16 *w_terms, int64_t T, int64_t E, int64_t H, int ks,
                                    float *logits, int *err, int sms, cudaStream_t s);
cudaError_t launch_x_to_f16(const __nv_bfloat16 *x, int64_t T, int64_t H, __half *x16, float *xscale,
                           cudaStream_t s);
size_t router_select_smem(int64_t E);
// queue: one int of device scratch (set to zero on the stream before the
// launch); warps take tokens from it.
cudaError_t launch_router_select(const __nv_bfloat16 *x, int64_t T, const float *W,
                                 const float *bias, int64_t E, int64_t H, int k,
                                 const float *logits, const float *wnorm, int ks, float gamma_d,
                                 int32_t *idx, float *wts, int32_t *queue, int *err, int sms,
                                 cudaStream_t s);

size_t permute_smem(int E);
// Chunks of the many-CTA sort for P pairs (chunk_hist needs chunks x E ints).
int64_t permute_chunks(int64_t P);
// Also clears pos_max[P] (if given) and the n_counters work counters.  With
// chunk_hist (device scratch of permute_chunks(P) x E ints) and more than two
// chunks the sort runs over many CTAs; otherwise in one CTA.
cudaError_t launch_permute(const int32_t *idx, int64_t P, int E, int tile_m, int32_t *counts,
                           int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *active,
                           int32_t *n_active, int32_t *tile_offsets, uint32_t *pos_max,
                           int32_t *counters, int n_counters, int *err, cudaStream_t s,
                           int32_t *chunk_hist = nullptr);

// Decode grouped GEMVs over the active experts' weight rows; T bounds the
// tokens any expert can hold (passes of 64 tokens above 64).
cudaError_t launch_gemv13(const uint8_t *w13, const float *s13, const __half *x16,
                          const float *xscale, const int32_t *counts, const int32_t *offsets,
                          const int32_t *perm, const int32_t *active, const int32_t *n_active,
                          int k, int64_t T, int64_t H, int64_t I, float *h, uint32_t *hmax,
                          int64_t max_items, int *err, int sms, cudaStream_t s,
                          const int32_t *slot_of = nullptr);
cudaError_t launch_gemv2(const uint8_t *w2, const float *s2, const float *h, const uint32_t *hmax,
                         const int32_t *counts, const int32_t *offsets, const int32_t *active,
                         const int32_t *n_active, int64_t T, int64_t H, int64_t I, float *y,
                         int64_t max_items, int *err, int sms, cudaStream_t s,
                         const int32_t *slot_of = nullptr);
bool encode_u8_tmap(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint32_t box_rows);
cudaError_t launch_act_quant(const __nv_bfloat16 *x, const int32_t *perm, int64_t P, int k,
                             int64_t H, int64_t Pmax, uint8_t *a_hi, uint8_t *a_lo, float *a_scale,
                             int sms, cudaStream_t s);
// Tensor maps of one grouped GEMM: up to three activation terms and the
// weights (loads), and the output boxes (stores): the three e4m3 terms of h
// (gate/up GEMM: boxes of 32 rows x 64 bytes) or y (down GEMM, st[0]: f32,
// boxes of 32 rows x 32 columns, 128-byte swizzle).
struct TmapSet {
  CUtensorMap a[3];
  CUtensorMap a64[3];  // the same activation terms in boxes of 64 rows (half tiles)
  CUtensorMap b;
  CUtensorMap st[3];
};
// Store maps of the grouped GEMM outputs (see TmapSet).
bool encode_h_store_tmap(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows);
bool encode_y_store_tmap(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows);
// mode 1: gate/up + SwiGLU -> three-term e4m3 h (two activation terms in);
// mode 2: down -> f32 y (three activation terms in).
// slot_of (here and in the other expert kernels): when given, expert e's
// weight codes are slab slot_of[e] of the weight tensors (an expert cache);
// its block scales stay at index e.
cudaError_t launch_grouped_gemm(int mode, const TmapSet &tm, const int32_t *offsets,
                                const int32_t *tile_offsets, const float *a_scale,
                                const float *w_scale, int E, int64_t H, int64_t I, int64_t Pmax,
                                uint8_t *const h_terms[3], float *h_scale, float *y, int *err,
                                int64_t max_items, int sms, cudaStream_t s,
                                const int32_t *slot_of = nullptr);
// Positions per tile of the tensor-core decode FFN.
constexpr int kDecodeTileN = 16;
// Tensor maps of the decode FFN: weights (W13 boxes of 128 rows, W2 boxes of
// 256 rows), the token-major x terms (boxes of one row, for tile::gather4) and
// the position-major h terms (boxes of kDecodeTileN rows).
struct DecodeMaps {
  CUtensorMap w13, w2;
  CUtensorMap x[2];
  CUtensorMap h[3];
};
// Gate/up + SwiGLU and down for small batches in one persistent launch
// (tile_offsets counted in tiles of kDecodeTileN positions).  x terms are
// token-major with scales x_scale[H/128][x_ld]; h is written as three e4m3
// terms with one power-of-two scale per (position, 128 outputs), h_scale
// [I/128][Pmax]; y f32 in three term planes [3][y_plane] of [P, H] (y of a
// pair is the sum of its three rows).  done13 [max_tiles + 1] (per-tile
// counters, then the work-queue head) must be zero on entry.
// Needs H % 256 == 0.
cudaError_t launch_decode_ffn(const DecodeMaps &maps, const int32_t *offsets,
                              const int32_t *tile_offsets, const int32_t *perm, int k,
                              const float *x_scale, int64_t x_ld, const float *s13, const float *s2,
                              int E, int64_t H, int64_t I, int64_t Pmax, uint8_t *const h_terms[3],
                              float *h_scale, float *y, int64_t y_plane, int32_t *done13, int *err,
                              int64_t max_tiles, int sms, cudaStream_t s,
                              const int32_t *slot_of = nullptr);
// Per-token activation terms (two e4m3 terms, one power-of-two scale per
// (token, 128 columns)); the token-major operand of the decode FFN.
cudaError_t launch_act_quant_tokens(const __nv_bfloat16 *x, int64_t T, int64_t H, uint8_t *a_hi,
                                    uint8_t *a_lo, float *a_scale, int64_t a_ld, int sms,
                                    cudaStream_t s);
// T <= 64 on the tensor-core decode path: logits and per-token activation
// terms, then (one CTA, chained by programmatic dependent launch) selection
// and the pair sort; counters [n_counters] are cleared.
float route_small_gamma(int64_t H, int64_t E);
cudaError_t launch_route_small(const __nv_bfloat16 *x, int64_t T, const float *W, const float *bias,
                               int64_t E, int64_t H, int k, float *logits, float *wnorm, float *xss,
                               uint8_t *a_hi, uint8_t *a_lo, float *a_scale, int64_t a_ld,
                               int32_t *counters, int n_counters, int32_t *idx,
                               float *wts, int32_t *counts, int32_t *offsets, int32_t *perm,
                               int32_t *inv, int32_t *active, int32_t *n_active,
                               int32_t *tile_offsets, int tile_m, int *err, cudaStream_t s);
// out[t] = sum_r wts[t, r] y[inv[t, r]], y of a pair being the sum of its rows
// in n_planes planes (stride plane) added in plane order.
cudaError_t launch_combine(const float *y, int n_planes, int64_t plane, const int32_t *inv,
                           const float *wts, int64_t T, int k, int64_t H, __nv_bfloat16 *out,
                           cudaStream_t s);

// FP4 (NVFP4) experts: grouped GEMVs with e2m1 codes [rows, K/2], e4m3 group
// scales [rows, K/16] and an f32 global scale per expert; h f32 [P, I] with
// per-position |h| maxima (hmax, cleared by the routing), y f32 [P, H].
cudaError_t launch_fp4_gate_up(const uint8_t *w13, const uint8_t *sf13, const float *g13,
                               const __half *x16, const float *xscale, const int32_t *counts,
                               const int32_t *offsets, const int32_t *perm, const int32_t *active,
                               const int32_t *n_active, int k, int64_t T, int64_t H, int64_t I,
                               float *h, uint32_t *hmax, int64_t max_items, int sms, cudaStream_t s);
cudaError_t launch_fp4_down(const uint8_t *w2, const uint8_t *sf2, const float *g2, const float *h,
                            const uint32_t *hmax, const int32_t *counts, const int32_t *offsets,
                            const int32_t *active, const int32_t *n_active, int64_t T, int64_t H,
                            int64_t I, float *y, int64_t max_items, int sms, cudaStream_t s);

// Decode attention (sub-block-1 of a shortcut-connected MoE layer): q bf16
// [B, n_heads, 128], K / V caches bf16 [B, S, n_kv_heads, 128], o bf16
// [B, n_heads, 128]; part: f32 workspace of B * n_heads * attention_chunks(S)
// * 130 floats.  n_heads / n_kv_heads in {1, 2, 4, 8}.
int64_t attention_chunks(int64_t S);
cudaError_t launch_decode_attention(const __nv_bfloat16 *q, const __nv_bfloat16 *kc,
                                    const __nv_bfloat16 *vc, int64_t B, int64_t S, int nh, int nkv,
                                    int d, float *part, __nv_bfloat16 *o, cudaStream_t s);

// One CTA whose waits (an mbarrier nothing arrives on, a global counter
// nothing increments) run out after limit_ns each: records DEV_ERR_TIMEOUT in
// *err and, if `which` is given, which waits gave up (bit 0 the mbarrier,
// bit 1 the counter).  *idle_counter must be 0 and stay 0.
cudaError_t launch_bounded_wait_selftest(const int32_t *idle_counter, uint64_t limit_ns, int *err,
                                         int32_t *which, cudaStream_t s);

}  // namespace fp8moe
