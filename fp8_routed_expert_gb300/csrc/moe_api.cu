// C ABI of the routed-MoE layer: context, workspace, argument checks and the
// order of kernel launches.  See include/fp8moe.h for the contract.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "fp8moe.h"
#include "common.cuh"
#include "ctx_internal.h"
#include "kernels.h"

using namespace fp8moe;

namespace {

constexpr int64_t kDecodeMaxT = 64;  // MOE_PATH_AUTO: tensor-core decode path up to this T

struct TimingRec {
  cudaEvent_t a, b;
  int kernel;
};

}  // namespace

struct moe_ctx {
  moe_config cfg{};
  int sms = 0;        // SMs the persistent kernels may use (moe_set_sm_budget)
  int sms_total = 0;  // SMs of the device
  char *ws = nullptr;
  size_t ws_bytes = 0;
  // workspace views
  float *logits = nullptr, *wnorm = nullptr, *wts = nullptr, *xscale = nullptr;
  float *h = nullptr, *y = nullptr;
  int32_t *idx = nullptr, *counts = nullptr, *offsets = nullptr, *perm = nullptr, *inv = nullptr;
  int32_t *active = nullptr, *n_active = nullptr, *tile_offsets = nullptr;
  int32_t *ticket = nullptr;  // completion ticket of the fused routing kernel (0 between calls)
  float *xnorm = nullptr;     // ||x_t||_2
  uint32_t *hmax = nullptr;
  __half *x16 = nullptr;
  __nv_bfloat16 *xin = nullptr, *xout = nullptr;  // staging for the host-buffer entry point
  uint8_t *a_hi = nullptr, *a_lo = nullptr, *h_t[3] = {nullptr, nullptr, nullptr};
  float *a_scale = nullptr;                      // [H/128][Pmax]
  float *h_scale = nullptr;                      // [I/128][Pmax] (GEMM) or [I/64][Pmax] (TCGEMV)
  TmapSet tm_gemm1, tm_gemm2;                    // activation terms (workspace) + last weights
  DecodeMaps dmaps;                              // tensor-core decode FFN operands
  float *xss = nullptr;                          // per-(token, 128 columns) sums of squares of x
  int32_t *done13 = nullptr;                     // decode FFN per-tile counters
  int32_t *chunk_hist = nullptr;                 // many-CTA pair sort: [chunks][E]
  int32_t *idle = nullptr;                       // a counter no kernel writes (bounded-wait self-test)
  __nv_bfloat16 *w_terms = nullptr;              // router W as three bf16 terms (large batches)
  CUtensorMap tm_rw, tm_rx;                      // maps of w_terms and of the last x
  const void *tm_rx_ptr = nullptr;               // x and T the map tm_rx describes
  int64_t tm_rx_T = 0;
  const void *tm_w13_ptr = nullptr, *tm_w2_ptr = nullptr;  // weights the maps in .b describe
  const void *dmaps_w13 = nullptr, *dmaps_w2 = nullptr;    // weights dmaps describe
  int *err = nullptr;
  int path = MOE_PATH_AUTO;
  // last forward
  int64_t last_T = 0;
  int last_k = 0;
  cudaStream_t last_stream = nullptr;
  // timing
  int timing = 0;  // bit mask of timed kernels
  int64_t n_launches = 0;
  std::vector<TimingRec> pending;
  std::vector<cudaEvent_t> spare;
  double total_ms[MOE_K_COUNT] = {};
  int64_t launches[MOE_K_COUNT] = {};
};

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

int check_config(const moe_config *c) {
  if (c->max_tokens <= 0 || c->hidden <= 0 || c->inter <= 0 || c->n_experts <= 0)
    return MOE_ERR_SHAPE;
  if (c->hidden % 128 != 0 || c->inter % 128 != 0) return MOE_ERR_SHAPE;
  if (c->hidden > 65536 || c->inter > 65536 || c->n_experts > 1024) return MOE_ERR_SHAPE;
  if (c->max_top_k < 1 || c->max_top_k > 32 || c->max_top_k > c->n_experts) return MOE_ERR_SHAPE;
  if (c->max_tokens > (int64_t)(INT32_MAX / 2) / c->max_top_k) return MOE_ERR_SHAPE;
  if (c->device < 0) return MOE_ERR_ARG;
  return MOE_OK;
}

// Events around one step's launches (n_kernels kernels) when timing is on.
struct Timed {
  moe_ctx *c;
  int kernel;
  cudaStream_t s;
  cudaEvent_t a = nullptr, b = nullptr;
  bool on;
  Timed(moe_ctx *ctx, int k, cudaStream_t st, int n_kernels = 1) : c(ctx), kernel(k), s(st) {
    c->n_launches += n_kernels;
    on = (c->timing >> k) & 1;
    if (!on) return;
    a = take();
    b = take();
    if (a) cudaEventRecord(a, s);
  }
  cudaEvent_t take() {
    if (!c->spare.empty()) {
      cudaEvent_t e = c->spare.back();
      c->spare.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
  }
  ~Timed() {
    if (!on || !a || !b) return;
    cudaEventRecord(b, s);
    c->pending.push_back({a, b, kernel});
  }
};

void drain_timing(moe_ctx *c) {
  for (auto &r : c->pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      c->total_ms[r.kernel] += ms;
      c->launches[r.kernel] += 1;
    }
    c->spare.push_back(r.a);
    c->spare.push_back(r.b);
  }
  c->pending.clear();
}

#define CUDA_TRY(expr)                          \
  do {                                          \
    cudaError_t e_ = (expr);                    \
    if (e_ != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

// The path a forward of T tokens takes.
int resolve_path(const moe_ctx *c, int64_t T) {
  int path = c->path != MOE_PATH_AUTO ? c->path : (T <= kDecodeMaxT ? MOE_PATH_TCGEMV : MOE_PATH_GEMM);
  // the tensor-core paths' down items are 256 output rows wide
  if ((path == MOE_PATH_GEMM || path == MOE_PATH_TCGEMV) && c->cfg.hidden % 256 != 0) path = MOE_PATH_GEMV;
  return path;
}

// Router logits of a large batch (T > kRouterWarpMaxT) on the tensor cores:
// row norms, the exact bf16 split of W, the logits in *ks planes; *gamma is
// the relative factor of their error bound.
int large_batch_logits(moe_ctx *c, const __nv_bfloat16 *x, int64_t T, const float *rw, int *ks,
                       float *gamma, cudaStream_t s) {
  const int64_t E = c->cfg.n_experts, H = c->cfg.hidden;
  *ks = router_tc_k_split(T, E, H, c->sms);
  *gamma = router_tc_gamma(H, *ks);
  if (c->tm_rx_ptr != x || c->tm_rx_T != T) {
    if (!encode_bf16_tmap(&c->tm_rx, x, H, T)) return MOE_ERR_CUDA;
    c->tm_rx_ptr = x;
    c->tm_rx_T = T;
  }
  Timed tm(c, MOE_K_ROUTER_LOGITS, s, 3);  // row norms, W split, logits
  CUDA_TRY(launch_row_norms(rw, E, H, c->wnorm, s));
  CUDA_TRY(launch_router_logits_tc(c->tm_rx, c->tm_rw, rw, c->w_terms, T, E, H, *ks, c->logits,
                                   c->err, c->sms, s));
  return MOE_OK;
}

// Routing for the grouped-GEMV and grouped-GEMM expert kernels: logits,
// certified top-k, the pair sort with 128-position tiles; for the GEMV
// kernels (gemv) also the f16 copy of x with its per-token power-of-two
// scale and cleared per-position |h| maxima.
int route_for_expert_kernels(moe_ctx *c, const __nv_bfloat16 *x, int64_t T, const float *rw,
                             const float *rb, int k, bool gemv, cudaStream_t s) {
  const int64_t E = c->cfg.n_experts, H = c->cfg.hidden, P = T * k;
  if (T <= kRouterWarpMaxT) {
    const float gamma = router_gamma(H);
    Timed tm(c, MOE_K_ROUTE, s);
    CUDA_TRY(launch_route_decode(x, T, rw, rb, E, H, k, gamma, c->logits, c->wnorm, c->xnorm,
                                 gemv ? c->x16 : nullptr, c->xscale, c->ticket, c->idx, c->wts,
                                 c->counts, c->offsets, c->perm, c->inv, c->active, c->n_active,
                                 c->tile_offsets, kTileM, gemv ? c->hmax : nullptr, c->err, s));
    return MOE_OK;
  }
  int ks = 1;
  float gamma = 0.f;
  {
    const int rc = large_batch_logits(c, x, T, rw, &ks, &gamma, s);
    if (rc != MOE_OK) return rc;
  }
  {
    Timed tm(c, MOE_K_ROUTER_SELECT, s);
    CUDA_TRY(launch_router_select(x, T, rw, rb, E, H, k, c->logits, c->wnorm, ks, gamma, c->idx,
                                  c->wts, c->ticket + 1, c->err, c->sms, s));
  }
  if (gemv) {
    c->n_launches += 1;
    CUDA_TRY(launch_x_to_f16(x, T, H, c->x16, c->xscale, s));
  }
  {
    Timed tm(c, MOE_K_PERMUTE, s, permute_chunks(P) > 2 ? 3 : 1);  // many-CTA sort above two chunks
    CUDA_TRY(launch_permute(c->idx, P, (int)E, kTileM, c->counts, c->offsets, c->perm, c->inv,
                            c->active, c->n_active, c->tile_offsets, gemv ? c->hmax : nullptr,
                            nullptr, 0, c->err, s, c->chunk_hist));
  }
  return MOE_OK;
}

// The layer with FP4 experts: routing as for the GEMV kernels, the two FP4
// grouped GEMVs, the rank-order combine.
int forward_nvfp4(moe_ctx *c, const __nv_bfloat16 *x, int64_t T, const float *rw, const float *rb,
                  const uint8_t *w13, const uint8_t *sf13, const float *g13, const uint8_t *w2,
                  const uint8_t *sf2, const float *g2, int k, __nv_bfloat16 *out, cudaStream_t s) {
  const int64_t E = c->cfg.n_experts, H = c->cfg.hidden, I = c->cfg.inter, P = T * k;
  const int64_t max_active = P < E ? P : E;
  if (T <= kRouterWarpMaxT) {
    // the two-kernel small-batch routing (it also clears the per-position
    // |h| maxima), then the f16 copy of x
    const int64_t Pm = c->cfg.max_tokens * c->cfg.max_top_k;
    {
      Timed tm(c, MOE_K_ROUTE, s, 2);
      CUDA_TRY(launch_route_small(x, T, rw, rb, E, H, k, c->logits, c->wnorm, c->xss, c->a_hi,
                                  c->a_lo, c->a_scale, Pm, reinterpret_cast<int32_t *>(c->hmax),
                                  (int)P, c->idx, c->wts, c->counts, c->offsets, c->perm, c->inv,
                                  c->active, c->n_active, c->tile_offsets, kTileM, c->err, s));
    }
    c->n_launches += 1;
    CUDA_TRY(launch_x_to_f16(x, T, H, c->x16, c->xscale, s));
  } else {
    const int rc = route_for_expert_kernels(c, x, T, rw, rb, k, true, s);
    if (rc != MOE_OK) return rc;
  }
  {
    Timed tm(c, MOE_K_GATE_UP, s);
    CUDA_TRY(launch_fp4_gate_up(w13, sf13, g13, c->x16, c->xscale, c->counts, c->offsets, c->perm,
                                c->active, c->n_active, k, T, H, I, c->h, c->hmax,
                                max_active * (I / 8), c->sms, s));
  }
  {
    Timed tm(c, MOE_K_DOWN, s);
    CUDA_TRY(launch_fp4_down(w2, sf2, g2, c->h, c->hmax, c->counts, c->offsets, c->active,
                             c->n_active, T, H, I, c->y, max_active * (H / 16), c->sms, s));
  }
  {
    Timed tm(c, MOE_K_COMBINE, s);
    CUDA_TRY(launch_combine(c->y, 1, 0, c->inv, c->wts, T, k, H, out, s));
  }
  c->last_T = T;
  c->last_k = k;
  c->last_stream = s;
  if (c->timing && c->pending.size() > 16384) drain_timing(c);
  return MOE_OK;
}

// Routing of the expert path `path`: everything before the expert kernels
// (for the tensor-core decode path also the activation terms).
int route_phase(moe_ctx *c, const __nv_bfloat16 *x, int64_t T, const float *rw, const float *rb,
                int k, int path, cudaStream_t s) {
  const int64_t E = c->cfg.n_experts, H = c->cfg.hidden;
  const int64_t P = T * k, Pm = c->cfg.max_tokens * c->cfg.max_top_k;
  const int64_t max_active = P < E ? P : E;
  if (path != MOE_PATH_TCGEMV) return route_for_expert_kernels(c, x, T, rw, rb, k, path == MOE_PATH_GEMV, s);
  const int64_t max_tiles = (P + kDecodeTileN - 1) / kDecodeTileN + max_active;
  if (T <= kRouterWarpMaxT) {
    Timed tm(c, MOE_K_ROUTE, s, 2);  // logits, then selection + sort
    CUDA_TRY(launch_route_small(x, T, rw, rb, E, H, k, c->logits, c->wnorm, c->xss, c->a_hi,
                                c->a_lo, c->a_scale, Pm, c->done13, (int)max_tiles + 1,
                                c->idx, c->wts, c->counts, c->offsets, c->perm, c->inv, c->active,
                                c->n_active, c->tile_offsets, kDecodeTileN, c->err, s));
    return MOE_OK;
  }
  int ks = 1;
  float gamma = 0.f;
  {
    const int rc = large_batch_logits(c, x, T, rw, &ks, &gamma, s);
    if (rc != MOE_OK) return rc;
  }
  {
    Timed tm(c, MOE_K_ROUTER_SELECT, s);
    CUDA_TRY(launch_router_select(x, T, rw, rb, E, H, k, c->logits, c->wnorm, ks, gamma, c->idx,
                                  c->wts, c->ticket + 1, c->err, c->sms, s));
  }
  {
    Timed tm(c, MOE_K_PERMUTE, s, permute_chunks(P) > 2 ? 3 : 1);  // many-CTA sort above two chunks
    CUDA_TRY(launch_permute(c->idx, P, (int)E, kDecodeTileN, c->counts, c->offsets, c->perm,
                            c->inv, c->active, c->n_active, c->tile_offsets, nullptr, c->done13,
                            (int)max_tiles + 1, c->err, s, c->chunk_hist));
  }
  {
    Timed tm(c, MOE_K_ACT_QUANT, s);
    CUDA_TRY(launch_act_quant_tokens(x, T, H, c->a_hi, c->a_lo, c->a_scale, Pm, c->sms, s));
  }
  return MOE_OK;
}

// The expert kernels of path `path` and the combine, on the routing that
// route_phase left in the context.
// slot_of / n_slabs: when slot_of is given, w13 and w2 hold n_slabs expert
// slabs and expert e's codes are slab slot_of[e] (an expert cache).
int expert_phase(moe_ctx *c, const __nv_bfloat16 *x, int64_t T, const uint8_t *w13,
                 const float *s13, const uint8_t *w2, const float *s2, int k, int path,
                 __nv_bfloat16 *out, cudaStream_t s, const int32_t *slot_of = nullptr,
                 int64_t n_slabs = 0) {
  const int64_t E = c->cfg.n_experts, H = c->cfg.hidden, I = c->cfg.inter;
  const int64_t NS = slot_of ? n_slabs : E;  // weight slabs the tensor maps cover
  const int64_t P = T * k, Pm = c->cfg.max_tokens * c->cfg.max_top_k;
  const int64_t max_active = P < E ? P : E;
  if (path == MOE_PATH_TCGEMV) {
    const int64_t max_tiles = (P + kDecodeTileN - 1) / kDecodeTileN + max_active;
    if (c->dmaps_w13 != w13) {
      if (!encode_u8_tmap(&c->dmaps.w13, w13, H, NS * 2 * I, 128)) return MOE_ERR_CUDA;
      c->dmaps_w13 = w13;
    }
    if (c->dmaps_w2 != w2) {
      if (!encode_u8_tmap(&c->dmaps.w2, w2, I, NS * H, 256)) return MOE_ERR_CUDA;
      c->dmaps_w2 = w2;
    }
    {
      Timed tm(c, MOE_K_GATE_UP, s);
      CUDA_TRY(launch_decode_ffn(c->dmaps, c->offsets, c->tile_offsets, c->perm, k, c->a_scale, Pm,
                                 s13, s2, (int)E, H, I, Pm, c->h_t, c->h_scale, c->y, P * H,
                                 c->done13, c->err, max_tiles, c->sms, s, slot_of));
    }
    {
      Timed tm(c, MOE_K_COMBINE, s);
      CUDA_TRY(launch_combine(c->y, 3, P * H, c->inv, c->wts, T, k, H, out, s));
    }
  } else {
    if (path == MOE_PATH_GEMV) {
      {
        Timed tm(c, MOE_K_GATE_UP, s);
        CUDA_TRY(launch_gemv13(w13, s13, c->x16, c->xscale, c->counts, c->offsets, c->perm,
                               c->active, c->n_active, k, T, H, I, c->h, c->hmax,
                               max_active * (I / 8), c->err, c->sms, s, slot_of));
      }
      {
        Timed tm(c, MOE_K_DOWN, s);
        CUDA_TRY(launch_gemv2(w2, s2, c->h, c->hmax, c->counts, c->offsets, c->active, c->n_active,
                              T, H, I, c->y, max_active * (H / 16), c->err, c->sms, s, slot_of));
      }
    } else {
      if (c->tm_w13_ptr != w13) {
        if (!encode_u8_tmap(&c->tm_gemm1.b, w13, H, NS * 2 * I, 64)) return MOE_ERR_CUDA;
        c->tm_w13_ptr = w13;
      }
      if (c->tm_w2_ptr != w2) {
        if (!encode_u8_tmap(&c->tm_gemm2.b, w2, I, NS * H, 64)) return MOE_ERR_CUDA;
        c->tm_w2_ptr = w2;
      }
      const int64_t max_tiles = (P + kTileM - 1) / kTileM + max_active;
      {
        Timed tm(c, MOE_K_ACT_QUANT, s);
        CUDA_TRY(launch_act_quant(x, c->perm, P, k, H, Pm, c->a_hi, c->a_lo, c->a_scale, c->sms, s));
      }
      {
        Timed tm(c, MOE_K_GATE_UP, s);
        CUDA_TRY(launch_grouped_gemm(1, c->tm_gemm1, c->offsets, c->tile_offsets, c->a_scale, s13,
                                     (int)E, H, I, Pm, c->h_t, c->h_scale, nullptr, c->err,
                                     max_tiles * (I / 128), c->sms, s, slot_of));
      }
      {
        Timed tm(c, MOE_K_DOWN, s);
        CUDA_TRY(launch_grouped_gemm(2, c->tm_gemm2, c->offsets, c->tile_offsets, c->h_scale, s2,
                                     (int)E, H, I, Pm, nullptr, nullptr, c->y, c->err,
                                     max_tiles * (H / 256), c->sms, s, slot_of));
      }
    }
    {
      Timed tm(c, MOE_K_COMBINE, s);
      CUDA_TRY(launch_combine(c->y, 1, 0, c->inv, c->wts, T, k, H, out, s));
    }
  }
  c->last_T = T;
  c->last_k = k;
  c->last_stream = s;
  if (c->timing && c->pending.size() > 16384) drain_timing(c);
  return MOE_OK;
}

int forward_device(moe_ctx *c, const __nv_bfloat16 *x, int64_t T, const float *rw,
                   const float *rb, const uint8_t *w13, const float *s13, const uint8_t *w2,
                   const float *s2, int k, __nv_bfloat16 *out, cudaStream_t s) {
  const int path = resolve_path(c, T);
  const int rc = route_phase(c, x, T, rw, rb, k, path, s);
  if (rc != MOE_OK) return rc;
  return expert_phase(c, x, T, w13, s13, w2, s2, k, path, out, s);
}

int check_forward_args(moe_ctx *c, const void *hidden, int64_t T, const float *rw,
                       const float *rb, const uint8_t *w13, const float *s13, const uint8_t *w2,
                       const float *s2, int32_t k, const void *out) {
  if (c == nullptr) return MOE_ERR_ARG;
  if (T < 0) return MOE_ERR_ARG;
  if (T > c->cfg.max_tokens) return MOE_ERR_SHAPE;
  if (k < 1 || k > c->cfg.max_top_k || k > c->cfg.n_experts) return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!hidden || !rw || !w13 || !s13 || !w2 || !s2 || !out) return MOE_ERR_ARG;
  if (!aligned(hidden, 16) || !aligned(rw, 16) || !aligned(w13, 16) || !aligned(w2, 16) ||
      !aligned(out, 16) || !aligned(s13, 4) || !aligned(s2, 4) || (rb && !aligned(rb, 4)))
    return MOE_ERR_ALIGN;
  return MOE_OK;
}

}  // namespace

namespace fp8moe {

int ctx_check_forward(moe_ctx *c, const void *hidden, int64_t T, const float *rw, const float *rb,
                      const uint8_t *w13, const float *s13, const uint8_t *w2, const float *s2,
                      int32_t k, const void *out, int *path) {
  const int rc = check_forward_args(c, hidden, T, rw, rb, w13, s13, w2, s2, k, out);
  if (rc == MOE_OK && path != nullptr) *path = resolve_path(c, T);
  return rc;
}

int ctx_route(moe_ctx *c, const __nv_bfloat16 *x, int64_t T, const float *rw, const float *rb,
              int k, int path, cudaStream_t s) {
  if (cudaSetDevice(c->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
  return route_phase(c, x, T, rw, rb, k, path, s);
}

int ctx_experts(moe_ctx *c, const __nv_bfloat16 *x, int64_t T, const uint8_t *w13,
                const float *s13, const uint8_t *w2, const float *s2, int k, int path,
                __nv_bfloat16 *out, cudaStream_t s, const int32_t *slot_of, int64_t n_slabs) {
  if (cudaSetDevice(c->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
  return expert_phase(c, x, T, w13, s13, w2, s2, k, path, out, s, slot_of, n_slabs);
}

int ctx_active_experts(moe_ctx *c, int32_t *buf, cudaStream_t s) {
  CUDA_TRY(cudaMemcpyAsync(buf, c->n_active, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaMemcpyAsync(buf + 1, c->active, (size_t)c->cfg.n_experts * sizeof(int32_t),
                           cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaStreamSynchronize(s));
  return MOE_OK;
}

const moe_config *ctx_config(const moe_ctx *c) { return &c->cfg; }

}  // namespace fp8moe

extern "C" {

const char *moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_SHAPE: return "unsupported shape (H, I multiples of 128; k in [1, min(E, max_top_k)]; T <= max_tokens)";
    case MOE_ERR_ALIGN: return "misaligned pointer";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait gave up";
    case MOE_ERR_NOMEM: return "workspace allocation failed";
    case MOE_ERR_UNSUPPORTED: return "device is not compute capability 10.3 (sm_103a)";
    case MOE_ERR_NONFINITE: return "a router logit was NaN or infinite";
    case MOE_ERR_DEVICE: return "device-side consistency check failed";
    default: return "unknown error";
  }
}

const char *moe_kernel_name(int kernel) {
  static const char *names[MOE_K_COUNT] = {"router_logits", "router_select", "permute",
                                           "gate_up_swiglu", "down", "combine", "act_quant",
                                           "route"};
  return (kernel >= 0 && kernel < MOE_K_COUNT) ? names[kernel] : "unknown";
}

int moe_init(moe_ctx **out, const moe_config *cfg) {
  if (out == nullptr) return MOE_ERR_ARG;
  *out = nullptr;
  if (cfg == nullptr) return MOE_ERR_ARG;
  int rc = check_config(cfg);
  if (rc != MOE_OK) return rc;

  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev <= 0) return MOE_ERR_CUDA;
  if (cfg->device >= ndev) return MOE_ERR_ARG;
  if (cudaSetDevice(cfg->device) != cudaSuccess) return MOE_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, cfg->device) != cudaSuccess) return MOE_ERR_CUDA;
  if (!(prop.major == 10 && prop.minor == 3)) return MOE_ERR_UNSUPPORTED;

  moe_ctx *c = new (std::nothrow) moe_ctx();
  if (c == nullptr) return MOE_ERR_NOMEM;
  c->cfg = *cfg;
  c->sms = prop.multiProcessorCount;
  c->sms_total = prop.multiProcessorCount;

  const int64_t Tm = cfg->max_tokens, E = cfg->n_experts, H = cfg->hidden, I = cfg->inter;
  const int64_t Pm = Tm * cfg->max_top_k;
  const int64_t Pr = (Pm + 127) / 128 * 128;  // rows of the GEMM operand buffers (whole 128-row boxes)
  struct Slot {
    void **p;
    size_t bytes;
  } slots[] = {
      {(void **)&c->logits, (size_t)(kRouterMaxKSplit * Tm * E) * 4},
      {(void **)&c->wnorm, (size_t)E * 4},
      {(void **)&c->idx, (size_t)Pm * 4},
      {(void **)&c->wts, (size_t)Pm * 4},
      {(void **)&c->counts, (size_t)E * 4},
      {(void **)&c->offsets, (size_t)(E + 1) * 4},
      {(void **)&c->perm, (size_t)Pm * 4},
      {(void **)&c->inv, (size_t)Pm * 4},
      {(void **)&c->active, (size_t)E * 4},
      {(void **)&c->n_active, 16},
      {(void **)&c->ticket, 16},
      {(void **)&c->idle, 16},
      {(void **)&c->w_terms, Tm > kRouterWarpMaxT ? (size_t)(3 * E * H) * 2 : 16},
      {(void **)&c->done13, (size_t)((Pm + kDecodeTileN - 1) / kDecodeTileN + E + 1) * 4},
      {(void **)&c->chunk_hist, (size_t)(permute_chunks(Pm) * E) * 4},
      {(void **)&c->xss, (size_t)(Tm * (H / 128)) * 4},
      {(void **)&c->xnorm, (size_t)Tm * 4},
      {(void **)&c->tile_offsets, (size_t)(E + 1) * 4},
      {(void **)&c->hmax, (size_t)Pm * 4},
      {(void **)&c->x16, (size_t)(Tm * H) * 2},
      {(void **)&c->xscale, (size_t)Tm * 4},
      {(void **)&c->h, (size_t)(Pm * I) * 4},
      {(void **)&c->y, (size_t)(3 * Pm * H) * 4},  // three term planes on the decode path
      {(void **)&c->xin, (size_t)(Tm * H) * 2},
      {(void **)&c->xout, (size_t)(Tm * H) * 2},
      {(void **)&c->err, 16},
      {(void **)&c->a_hi, (size_t)(Pr * H)},
      {(void **)&c->a_lo, (size_t)(Pr * H)},
      {(void **)&c->a_scale, (size_t)(H / 128 * Pm) * 4},
      {(void **)&c->h_t[0], (size_t)(Pr * I)},
      {(void **)&c->h_t[1], (size_t)(Pr * I)},
      {(void **)&c->h_t[2], (size_t)(Pr * I)},
      {(void **)&c->h_scale, (size_t)(I / 64 * Pm) * 4},
  };
  size_t total = 0;
  for (auto &s : slots) total += align_up(s.bytes, 256);
  if (cudaMalloc(&c->ws, total) != cudaSuccess) {
    cudaGetLastError();
    delete c;
    return MOE_ERR_NOMEM;
  }
  c->ws_bytes = total;
  size_t off = 0;
  for (auto &s : slots) {
    *s.p = c->ws + off;
    off += align_up(s.bytes, 256);
  }
  if (cudaMemset(c->ws, 0, total) != cudaSuccess) {
    cudaFree(c->ws);
    delete c;
    return MOE_ERR_CUDA;
  }
  if ((Tm > kRouterWarpMaxT && !encode_bf16_tmap(&c->tm_rw, c->w_terms, H, 3 * E)) ||
      !encode_u8_tmap(&c->tm_gemm1.a[0], c->a_hi, H, Pr, 128) ||
      !encode_u8_tmap(&c->tm_gemm1.a[1], c->a_lo, H, Pr, 128) ||
      !encode_u8_tmap(&c->tm_gemm1.a[2], c->a_lo, H, Pr, 128) ||
      !encode_u8_tmap(&c->tm_gemm2.a[0], c->h_t[0], I, Pr, 128) ||
      !encode_u8_tmap(&c->tm_gemm2.a[1], c->h_t[1], I, Pr, 128) ||
      !encode_u8_tmap(&c->tm_gemm2.a[2], c->h_t[2], I, Pr, 128) ||
      !encode_u8_tmap(&c->tm_gemm1.a64[0], c->a_hi, H, Pr, 64) ||
      !encode_u8_tmap(&c->tm_gemm1.a64[1], c->a_lo, H, Pr, 64) ||
      !encode_u8_tmap(&c->tm_gemm1.a64[2], c->a_lo, H, Pr, 64) ||
      !encode_u8_tmap(&c->tm_gemm2.a64[0], c->h_t[0], I, Pr, 64) ||
      !encode_u8_tmap(&c->tm_gemm2.a64[1], c->h_t[1], I, Pr, 64) ||
      !encode_u8_tmap(&c->tm_gemm2.a64[2], c->h_t[2], I, Pr, 64) ||
      !encode_h_store_tmap(&c->tm_gemm1.st[0], c->h_t[0], I, Pr) ||
      !encode_h_store_tmap(&c->tm_gemm1.st[1], c->h_t[1], I, Pr) ||
      !encode_h_store_tmap(&c->tm_gemm1.st[2], c->h_t[2], I, Pr) ||
      !encode_y_store_tmap(&c->tm_gemm2.st[0], c->y, H, Pm) ||
      !encode_u8_tmap(&c->dmaps.x[0], c->a_hi, H, Tm, 1) ||
      !encode_u8_tmap(&c->dmaps.x[1], c->a_lo, H, Tm, 1) ||
      !encode_u8_tmap(&c->dmaps.h[0], c->h_t[0], I, Pr, kDecodeTileN) ||
      !encode_u8_tmap(&c->dmaps.h[1], c->h_t[1], I, Pr, kDecodeTileN) ||
      !encode_u8_tmap(&c->dmaps.h[2], c->h_t[2], I, Pr, kDecodeTileN)) {
    cudaFree(c->ws);
    delete c;
    return MOE_ERR_CUDA;
  }
  *out = c;
  return MOE_OK;
}

void moe_free(moe_ctx *c) {
  if (c == nullptr) return;
  cudaSetDevice(c->cfg.device);
  drain_timing(c);
  for (auto e : c->spare) cudaEventDestroy(e);
  if (c->ws) cudaFree(c->ws);
  delete c;
}

int moe_layer_forward(moe_ctx *c, const void *hidden, int64_t T, const float *rw,
                      const float *rb, const uint8_t *w13, const float *s13, const uint8_t *w2,
                      const float *s2, int32_t top_k, void *out, void *stream) {
  int rc = check_forward_args(c, hidden, T, rw, rb, w13, s13, w2, s2, top_k, out);
  if (rc != MOE_OK) return rc;
  if (T == 0) {
    c->last_T = 0;
    c->last_k = top_k;
    return MOE_OK;
  }
  if (cudaSetDevice(c->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
  return forward_device(c, (const __nv_bfloat16 *)hidden, T, rw, rb, w13, s13, w2, s2, top_k,
                        (__nv_bfloat16 *)out, (cudaStream_t)stream);
}

int moe_layer_forward_nvfp4(moe_ctx *c, const void *hidden, int64_t T, const float *rw,
                            const float *rb, const uint8_t *w13, const uint8_t *sf13,
                            const float *g13, const uint8_t *w2, const uint8_t *sf2,
                            const float *g2, int32_t top_k, void *out, void *stream) {
  // shapes, T and k as for the FP8 entry point (the scale arguments are
  // checked there for 4-byte alignment; here the group scales need 2)
  int rc = check_forward_args(c, hidden, T, rw, rb, w13, g13, w2, g2, top_k, out);
  if (rc != MOE_OK) return rc;
  if (T == 0) {
    c->last_T = 0;
    c->last_k = top_k;
    return MOE_OK;
  }
  if (!sf13 || !sf2) return MOE_ERR_ARG;
  if (!aligned(sf13, 2) || !aligned(sf2, 2)) return MOE_ERR_ALIGN;
  if (cudaSetDevice(c->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
  return forward_nvfp4(c, (const __nv_bfloat16 *)hidden, T, rw, rb, w13, sf13, g13, w2, sf2, g2,
                       top_k, (__nv_bfloat16 *)out, (cudaStream_t)stream);
}

int moe_layer_forward_host(moe_ctx *c, const void *hidden_host, int64_t T, const float *rw,
                           const float *rb, const uint8_t *w13, const float *s13,
                           const uint8_t *w2, const float *s2, int32_t top_k, void *out_host,
                           void *stream) {
  if (c == nullptr) return MOE_ERR_ARG;
  int rc = check_forward_args(c, c->xin, T, rw, rb, w13, s13, w2, s2, top_k, c->xout);
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (!hidden_host || !out_host) return MOE_ERR_ARG;
  if (cudaSetDevice(c->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t bytes = (size_t)(T * c->cfg.hidden) * 2;
  CUDA_TRY(cudaMemcpyAsync(c->xin, hidden_host, bytes, cudaMemcpyHostToDevice, s));
  rc = forward_device(c, c->xin, T, rw, rb, w13, s13, w2, s2, top_k, c->xout, s);
  if (rc != MOE_OK) return rc;
  CUDA_TRY(cudaMemcpyAsync(out_host, c->xout, bytes, cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaStreamSynchronize(s));
  return MOE_OK;
}

int moe_get_routing(moe_ctx *c, int32_t *idx, float *wts, int32_t *counts, int32_t *offsets,
                    int32_t *perm, int32_t *inv, void *stream) {
  if (c == nullptr) return MOE_ERR_ARG;
  if (cudaSetDevice(c->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t P = (size_t)(c->last_T * c->last_k), E = (size_t)c->cfg.n_experts;
  const cudaMemcpyKind d2d = cudaMemcpyDeviceToDevice;
  if (idx && P) CUDA_TRY(cudaMemcpyAsync(idx, c->idx, P * 4, d2d, s));
  if (wts && P) CUDA_TRY(cudaMemcpyAsync(wts, c->wts, P * 4, d2d, s));
  if (counts) CUDA_TRY(cudaMemcpyAsync(counts, c->counts, E * 4, d2d, s));
  if (offsets) CUDA_TRY(cudaMemcpyAsync(offsets, c->offsets, (E + 1) * 4, d2d, s));
  if (perm && P) CUDA_TRY(cudaMemcpyAsync(perm, c->perm, P * 4, d2d, s));
  if (inv && P) CUDA_TRY(cudaMemcpyAsync(inv, c->inv, P * 4, d2d, s));
  return MOE_OK;
}

int moe_status(moe_ctx *c) {
  if (c == nullptr) return MOE_ERR_ARG;
  if (cudaSetDevice(c->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(c->last_stream) != cudaSuccess) return MOE_ERR_CUDA;
  int flag = 0;
  CUDA_TRY(cudaMemcpy(&flag, c->err, sizeof(int), cudaMemcpyDeviceToHost));
  CUDA_TRY(cudaMemset(c->err, 0, sizeof(int)));
  if (flag & DEV_ERR_TIMEOUT) return MOE_ERR_DEVICE_TIMEOUT;
  if (flag & DEV_ERR_NONFINITE) return MOE_ERR_NONFINITE;
  if (flag) return MOE_ERR_DEVICE;
  return MOE_OK;
}

int moe_selftest_wait_timeout(moe_ctx *c, int64_t limit_ns, int32_t *which, void *stream) {
  if (c == nullptr || limit_ns <= 0 || limit_ns > 1000000000ll) return MOE_ERR_ARG;
  if (which != nullptr && !aligned(which, 4)) return MOE_ERR_ALIGN;
  if (cudaSetDevice(c->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  c->n_launches += 1;
  CUDA_TRY(launch_bounded_wait_selftest(c->idle, (uint64_t)limit_ns, c->err, which, s));
  c->last_stream = s;
  return MOE_OK;
}

int moe_set_sm_budget(moe_ctx *c, int32_t n_sms) {
  if (c == nullptr) return MOE_ERR_ARG;
  c->sms = (n_sms <= 0 || n_sms > c->sms_total) ? c->sms_total : n_sms;
  return MOE_OK;
}

int64_t moe_attention_workspace_bytes(int64_t B, int64_t S, int32_t n_heads, int32_t head_dim) {
  if (B < 0 || S < 1 || n_heads < 1 || head_dim < 1) return MOE_ERR_ARG;
  return B * n_heads * attention_chunks(S) * (head_dim + 2) * (int64_t)sizeof(float);
}

int moe_decode_attention(const void *q, const void *k_cache, const void *v_cache, int64_t B,
                         int64_t S, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, void *out,
                         void *workspace, int64_t workspace_bytes, void *stream) {
  if (B < 0 || S < 1) return MOE_ERR_ARG;
  if (head_dim != 128 || n_kv_heads < 1 || n_heads < n_kv_heads || n_heads % n_kv_heads != 0)
    return MOE_ERR_SHAPE;
  const int g = n_heads / n_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return MOE_ERR_SHAPE;
  if (B > 65535 || n_kv_heads > 65535 || attention_chunks(S) > INT32_MAX) return MOE_ERR_SHAPE;
  if (B == 0) return MOE_OK;
  if (!q || !k_cache || !v_cache || !out || !workspace) return MOE_ERR_ARG;
  if (workspace_bytes < moe_attention_workspace_bytes(B, S, n_heads, head_dim)) return MOE_ERR_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(workspace, 16))
    return MOE_ERR_ALIGN;
  CUDA_TRY(launch_decode_attention(static_cast<const __nv_bfloat16 *>(q),
                                   static_cast<const __nv_bfloat16 *>(k_cache),
                                   static_cast<const __nv_bfloat16 *>(v_cache), B, S, n_heads,
                                   n_kv_heads, head_dim, static_cast<float *>(workspace),
                                   static_cast<__nv_bfloat16 *>(out), static_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

int moe_set_path(moe_ctx *c, int path) {
  if (c == nullptr) return MOE_ERR_ARG;
  if (path != MOE_PATH_AUTO && path != MOE_PATH_GEMV && path != MOE_PATH_GEMM &&
      path != MOE_PATH_TCGEMV)
    return MOE_ERR_ARG;
  c->path = path;
  return MOE_OK;
}

int moe_resolve_path(moe_ctx *c, int64_t T) {
  if (c == nullptr || T < 0) return MOE_ERR_ARG;
  return resolve_path(c, T);
}

int moe_set_timing(moe_ctx *c, int mask) {
  if (c == nullptr) return MOE_ERR_ARG;
  if (cudaSetDevice(c->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
  drain_timing(c);
  for (int k = 0; k < MOE_K_COUNT; ++k) {
    c->total_ms[k] = 0.0;
    c->launches[k] = 0;
  }
  c->timing = mask & ((1 << MOE_K_COUNT) - 1);
  return MOE_OK;
}

int64_t moe_launch_count(moe_ctx *c) { return c ? c->n_launches : -1; }

int moe_kernel_time(moe_ctx *c, int kernel, double *total_ms, int64_t *launches) {
  if (c == nullptr || kernel < 0 || kernel >= MOE_K_COUNT) return MOE_ERR_ARG;
  if (cudaSetDevice(c->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
  drain_timing(c);
  if (total_ms) *total_ms = c->total_ms[kernel];
  if (launches) *launches = c->launches[kernel];
  return MOE_OK;
}

int moe_debug_copy(moe_ctx *c, const char *name, void *dst, int64_t capacity, int64_t *nbytes,
                   void *stream) {
  if (c == nullptr || name == nullptr || capacity < 0) return MOE_ERR_ARG;
  const int64_t T = c->last_T, P = c->last_T * c->last_k;
  const int64_t E = c->cfg.n_experts, H = c->cfg.hidden, I = c->cfg.inter;
  const void *p = nullptr;
  int64_t n = 0;
  if (!strcmp(name, "logits")) { p = c->logits; n = T * E * 4; }
  else if (!strcmp(name, "h")) { p = c->h; n = P * I * 4; }
  else if (!strcmp(name, "y")) { p = c->y; n = P * H * 4; }
  else if (!strcmp(name, "y_terms")) { p = c->y; n = 3 * P * H * 4; }
  else if (!strcmp(name, "x16")) { p = c->x16; n = T * H * 2; }
  else return MOE_ERR_ARG;
  if (nbytes) *nbytes = n;
  const int64_t m = n < capacity ? n : capacity;
  if (m > 0) {
    if (dst == nullptr) return MOE_ERR_ARG;
    if (cudaSetDevice(c->cfg.device) != cudaSuccess) return MOE_ERR_CUDA;
    CUDA_TRY(cudaMemcpyAsync(dst, p, (size_t)m, cudaMemcpyDeviceToDevice, (cudaStream_t)stream));
  }
  return MOE_OK;
}

}  // extern "C"
