/*
 * fp8moe.h - C ABI of a GB300 (sm_103a) routed Mixture-of-Experts FFN layer
 * whose expert weights are blockwise FP8.
 *
 * The layer (one decoder MoE block's routed experts) computes, for T tokens:
 *   1. router logits in f32 inputs (dragon.c, "Precision": router f32),
 *      top-k by logit with ties to the lower expert index (Trochilus, "What
 *      makes it different", the lowest row wins a tie), weights = softmax over
 *      the k selected logits (softmax, top-k, renormalise);
 *   2. a histogram / exclusive scan / stable scatter of the T*k (token,
 *      expert) pairs by expert (Trochilus, "Acknowledgements": pairs sorted by
 *      a counting sort);
 *   3. per expert, SwiGLU: h = silu(W13[e, :I] x) * (W13[e, I:] x), with the
 *      gate rows before the up rows (DeepSeek-V4.1-Flash post, "Repack experts
 *      for the disk": gate | up | down);
 *   4. y = W2[e] h;
 *   5. out[t] = bf16( sum over r = 0..k-1, in router rank order, of
 *      w[t, r] * y[t, r] ) (WARP BACKENDS.md, "Coherent memory": partials
 *      reduced in original router order), with no float atomics.
 * Weights are e4m3 codes with one f32 scale per 128x128 block, stored with
 * the weights (dragon.c, "Precision"); a weight's value is its code's value
 * times its block's scale.
 *
 * Conventions (every call):
 *   - Return value: MOE_OK (0) or a negative MOE_ERR_* code; nothing throws.
 *   - Tensor arguments are raw pointers; "device" pointers must be CUDA
 *     device (or managed) memory of the context's device.  The caller owns
 *     every tensor; the context owns only its workspace.
 *   - All integer sizes are int64_t; all index arithmetic inside is 64-bit.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the host is not synchronised, except where stated.
 *   - One context serves one stream at a time: calls on one context must not
 *     overlap on the GPU.
 */
#ifndef FP8MOE_H
#define FP8MOE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_ARG (-1)            /* NULL pointer, bad enum, T < 0          */
#define MOE_ERR_SHAPE (-2)          /* H or I not a multiple of 128, k out of  */
                                    /* [1, min(E, max_top_k)], T > max_tokens  */
#define MOE_ERR_ALIGN (-3)          /* a pointer breaks its stated alignment   */
#define MOE_ERR_CUDA (-4)           /* a CUDA runtime/driver call failed       */
#define MOE_ERR_DEVICE_TIMEOUT (-5) /* a bounded device-side wait gave up      */
#define MOE_ERR_NOMEM (-6)          /* workspace allocation failed             */
#define MOE_ERR_UNSUPPORTED (-7)    /* device is not compute capability 10.3   */
#define MOE_ERR_NONFINITE (-8)      /* a router logit was NaN or infinite      */
#define MOE_ERR_DEVICE (-9)         /* a device-side consistency check failed  */

typedef struct moe_ctx moe_ctx; /* opaque; owned by the library */

typedef struct moe_config {
  int64_t max_tokens; /* largest T a forward may be called with (> 0)            */
  int64_t hidden;     /* H: model width, multiple of 128, <= 65536              */
  int64_t n_experts;  /* E: routed experts, 1..1024                             */
  int64_t inter;      /* I: expert FFN width, multiple of 128, <= 65536         */
  int32_t max_top_k;  /* largest k a forward may use, 1..min(E, 32)             */
  int32_t device;     /* CUDA device ordinal the context lives on              */
} moe_config;

/*
 * moe_init - validate `cfg` and allocate a context with a device workspace
 * sized for max_tokens * max_top_k (token, expert) pairs.
 *   out : receives the new context (host pointer to a host pointer).
 * Errors: MOE_ERR_ARG (NULL), MOE_ERR_SHAPE (cfg out of range; checked before
 * any CUDA call), MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_NOMEM.  On error
 * *out is set to NULL and nothing is leaked.
 */
int moe_init(moe_ctx **out, const moe_config *cfg);

/*
 * moe_layer_forward - run the layer on T tokens (steps 1-5 above).
 *   hidden      : device, bf16 [T, H] row-major, 16-byte aligned.
 *   router_w    : device, f32 [E, H] row-major, 16-byte aligned.
 *   router_bias : device, f32 [E], or NULL for none.  When present it is added
 *                 to the logits before selection and softmax.
 *   w13         : device, e4m3 [E, 2I, H] row-major (rows [0,I) gate,
 *                 [I,2I) up), 16-byte aligned.
 *   s13         : device, f32 [E, 2I/128, H/128] block scales, 4-byte aligned.
 *   w2          : device, e4m3 [E, H, I] row-major, 16-byte aligned.
 *   s2          : device, f32 [E, H/128, I/128] block scales, 4-byte aligned.
 *   top_k       : k, in [1, min(E, max_top_k)].
 *   out         : device, bf16 [T, H], 16-byte aligned; must not overlap any
 *                 input.
 *   stream      : cudaStream_t or NULL.
 * T = 0 is a no-op.  Routing is exact: indices, counts and the permutation
 * equal those of exact arithmetic on the inputs (f32 logits carry a rigorous
 * error bound; tokens whose order the bound cannot certify are recomputed
 * from exact products with every rounding error carried).  Device-side failures (a bounded wait that gave up, a non-finite
 * logit) are recorded in the context and reported by moe_status.
 */
int moe_layer_forward(moe_ctx *ctx, const void *hidden, int64_t T, const float *router_w,
                      const float *router_bias, const uint8_t *w13, const float *s13,
                      const uint8_t *w2, const float *s2, int32_t top_k, void *out,
                      void *stream);

/*
 * moe_layer_forward_host - moe_layer_forward with the activations in HOST
 * memory: copies hidden_host (bf16 [T, H]) to the device, runs the layer, and
 * copies the result into out_host (bf16 [T, H]).  Weights stay device
 * pointers as in moe_layer_forward.  Host buffers should be pinned
 * (cudaHostAlloc / cudaHostRegister) for asynchronous copies.  The call
 * returns after the result is in out_host (it synchronises `stream`).
 */
int moe_layer_forward_host(moe_ctx *ctx, const void *hidden_host, int64_t T,
                           const float *router_w, const float *router_bias, const uint8_t *w13,
                           const float *s13, const uint8_t *w2, const float *s2, int32_t top_k,
                           void *out_host, void *stream);

/*
 * moe_layer_forward_nvfp4 - the same layer (steps 1-5 above) with FP4 expert
 * weights in the NVFP4 format of the Qwen post's experts ("Why this model, of
 * all models"; "The engine", piece 1: half a byte per weight plus one e4m3
 * scale per 16 weights; piece 4: the e2m1 -> f16x2 hardware conversion).  A
 * weight's value is e2m1(code) * e4m3(group scale) * global scale.  The
 * router, hidden, out, top_k and stream arguments are those of
 * moe_layer_forward.
 *   w13  : device, u8 [E, 2I, H/2]: e2m1 codes of W13 (rows [0,I) gate,
 *          [I,2I) up), two per byte along H, element 2j in the low nibble;
 *          16-byte aligned.
 *   sf13 : device, u8 [E, 2I, H/16]: e4m3 scale of each 16 consecutive
 *          weights of a row; 2-byte aligned.
 *   g13  : device, f32 [E]: global scale of each expert's W13; 4-byte aligned.
 *   w2, sf2, g2 : the same for W2 [E, H, I] (codes [E, H, I/2], scales
 *          [E, H, I/16], globals [E]).
 * The expert kernels are grouped GEMVs (any T; built for small batches).
 * Errors as for moe_layer_forward; sf13 / sf2 NULL is MOE_ERR_ARG.
 */
int moe_layer_forward_nvfp4(moe_ctx *ctx, const void *hidden, int64_t T, const float *router_w,
                            const float *router_bias, const uint8_t *w13, const uint8_t *sf13,
                            const float *g13, const uint8_t *w2, const uint8_t *sf2,
                            const float *g2, int32_t top_k, void *out, void *stream);

/*
 * moe_get_routing - copy the routing of the last forward into caller device
 * buffers (any may be NULL to skip it).  Sizes for that forward's T and k,
 * P = T*k:
 *   idx     int32 [T, k]  experts of each token in rank order
 *   wts     f32   [T, k]  renormalised weights, same order
 *   counts  int32 [E]     pairs routed to each expert
 *   offsets int32 [E+1]   exclusive scan of counts
 *   perm    int32 [P]     position -> pair id p = t*k + r, ascending p within
 *                         each expert segment
 *   inv     int32 [P]     pair id -> position
 * Enqueued on `stream`.
 */
int moe_get_routing(moe_ctx *ctx, int32_t *idx, float *wts, int32_t *counts, int32_t *offsets,
                    int32_t *perm, int32_t *inv, void *stream);

/*
 * moe_status - synchronise the context's last stream and return MOE_OK or
 * the first device-side error recorded since the previous call (the flag is
 * cleared).
 */
int moe_status(moe_ctx *ctx);

/* moe_free - release the context and its workspace; NULL is a no-op. */
void moe_free(moe_ctx *ctx);

/* moe_strerror - static description of a return code. */
const char *moe_strerror(int code);

/*
 * Path selection.  MOE_PATH_AUTO picks the tensor-core decode path for
 * T <= 64 and the tensor-core grouped-GEMM path above (both need H % 256 == 0;
 * otherwise the grouped-GEMV path runs); the other values force one path (all
 * compute the same layer).
 *   MOE_PATH_GEMV   e4m3 weights dequantised in registers, mma.sync f16
 *                   (activations as f16 hi/lo pairs);
 *   MOE_PATH_GEMM   tcgen05 grouped GEMM, tiles of 128 positions;
 *   MOE_PATH_TCGEMV tcgen05 decode FFN: gate/up and down in one launch, tiles
 *                   of 16 positions (the weight rows are the MMA's N operand).
 */
#define MOE_PATH_AUTO 0
#define MOE_PATH_GEMV 1
#define MOE_PATH_GEMM 2
#define MOE_PATH_TCGEMV 3
int moe_set_path(moe_ctx *ctx, int path);
/* moe_resolve_path - the MOE_PATH_* (not AUTO) a forward of T tokens would
 * take on this context; MOE_ERR_ARG for a NULL context or T < 0. */
int moe_resolve_path(moe_ctx *ctx, int64_t T);

/*
 * Kernel timing.  moe_set_timing(ctx, mask) records CUDA events around each
 * kernel whose bit (1 << MOE_K_*) is set in `mask`, on the forward's stream
 * (mask 0 turns timing off; every call resets the totals).  moe_kernel_time
 * returns the summed device time (ms) and the number of timed launches of one
 * kernel (it synchronises).  moe_launch_count returns how many kernels the
 * context has launched since moe_init, timed or not.
 */
#define MOE_K_ROUTER_LOGITS 0
#define MOE_K_ROUTER_SELECT 1
#define MOE_K_PERMUTE 2
#define MOE_K_GATE_UP 3 /* grouped GEMV or GEMM for W13 with SwiGLU */
#define MOE_K_DOWN 4    /* grouped GEMV or GEMM for W2            */
#define MOE_K_COMBINE 5
#define MOE_K_ACT_QUANT 6
#define MOE_K_ROUTE 7   /* small batches: logits, selection and sort in one kernel */
#define MOE_K_COUNT 8
int moe_set_timing(moe_ctx *ctx, int mask);
int moe_kernel_time(moe_ctx *ctx, int kernel, double *total_ms, int64_t *launches);
int64_t moe_launch_count(moe_ctx *ctx);
const char *moe_kernel_name(int kernel);

/*
 * moe_debug_copy - copy a workspace buffer of the last forward into a caller
 * device buffer, for tests: "logits" f32 [T,E], "h" f32 [P,I] (GEMV path,
 * position order), "y" f32 [P,H] (position order; GEMV and GEMM paths),
 * "y_terms" f32 [3,P,H] (tensor-core decode path: y of a position is the sum
 * of its three rows, one per h term), "x16" f16 [T,H].  Copies
 * min(capacity, size) bytes on `stream` and stores the buffer's full size in
 * *nbytes (may be NULL).
 */
int moe_debug_copy(moe_ctx *ctx, const char *name, void *dst, int64_t capacity, int64_t *nbytes,
                   void *stream);

/*
 * Experts larger than device memory (DeepSeek-V4.1-Flash post, "Bytes per
 * token decide everything" and "Making it faster", v4: a cache in front of
 * the slow tier and the next layer's experts guessed from its router and
 * prefetched into the gap; Qwen post, "Where the time actually goes":
 * speculative copies one layer early).  The expert weights (e4m3 codes) stay
 * in host memory; `n_slots` experts at a time are held in device memory
 * (slabs of one expert's W13 and W2 codes) and streamed in over NVLink-C2C;
 * the layer's own kernels read expert e's codes from the slab a table names.
 * The f32 block scales (1/16384 of the codes) stay resident and are passed
 * as device pointers.
 *
 * moe_cache_init - create a cache for context `ctx`.
 *   w13_host : host, e4m3 [E, 2I, H] (layout of moe_layer_forward's w13).
 *   w2_host  : host, e4m3 [E, H, I].
 *   n_slots  : experts held in device memory, 1..E (3*I*H bytes of device
 *              memory each).
 * The host ranges are page-locked (cudaHostRegister) for the life of the
 * cache unless the caller already registered them; they must stay valid and
 * unchanged until moe_cache_free.
 * Errors: MOE_ERR_ARG, MOE_ERR_SHAPE (n_slots out of range), MOE_ERR_NOMEM,
 * MOE_ERR_CUDA.
 */
typedef struct moe_expert_cache moe_expert_cache;
int moe_cache_init(moe_expert_cache **out, moe_ctx *ctx, const uint8_t *w13_host,
                   const uint8_t *w2_host, int64_t n_slots);

/*
 * moe_cache_forward - moe_layer_forward with the cache's experts: routes on
 * `stream`, waits for the active-expert list (a host synchronisation of
 * `stream`), brings the missing experts into least recently used slots
 * (copies on `stream`), waits for earlier prefetches, then enqueues the
 * expert kernels and the combine.  Results are bit-identical to
 * moe_layer_forward with the same weights in device memory.  Consecutive
 * forwards of one cache must use one stream.  MOE_ERR_NOMEM if the batch
 * needs more experts than there are slots.
 */
int moe_cache_forward(moe_expert_cache *c, const void *hidden, int64_t T, const float *router_w,
                      const float *router_bias, const float *s13, const float *s2, int32_t top_k,
                      void *out, void *stream);

/*
 * moe_cache_prefetch - start bringing `experts` (host array of n expert
 * ids, best guess first) into the cache on the cache's own copy stream,
 * into slots that the last forward does not use; stops when no such slot is
 * left.  Returns the number of copies started (>= 0) or an error.  The next
 * moe_cache_forward waits for them.
 */
int moe_cache_prefetch(moe_expert_cache *c, const int32_t *experts, int64_t n);

/*
 * moe_cache_guess - the experts a router would pick for `hidden`: routes
 * hidden (device bf16 [T, H], T <= 64) with router_w / router_bias (device,
 * f32 [E, H] / [E] or NULL) on the cache's own stream, and writes to
 * experts_out (host, n_guess ints) the chosen experts ordered by the number
 * of tokens choosing them, then by their best rank, then by id.  Used with
 * the NEXT layer's router on this layer's input to guess what to prefetch.
 * Returns the number written (<= n_guess) or an error.
 */
int moe_cache_guess(moe_expert_cache *c, const void *hidden, int64_t T, const float *router_w,
                    const float *router_bias, int32_t top_k, int32_t n_guess, int32_t *experts_out);

/* moe_cache_stats - counters since moe_cache_init, out[0 .. n-1] (host). */
#define MOE_CACHE_HITS 0          /* active experts found in the cache        */
#define MOE_CACHE_MISSES 1        /* active experts copied in by a forward    */
#define MOE_CACHE_PREFETCHED 2    /* experts copied in by moe_cache_prefetch  */
#define MOE_CACHE_PREFETCH_USED 3 /* prefetched experts a forward then used   */
#define MOE_CACHE_EVICTIONS 4
#define MOE_CACHE_BYTES_COPIED 5  /* host -> device bytes of expert codes     */
#define MOE_CACHE_STATS 6
int moe_cache_stats(const moe_expert_cache *c, int64_t *out, int32_t n);

/* moe_cache_resident - slot of every expert, -1 if not cached (host int[E]). */
int moe_cache_resident(const moe_expert_cache *c, int32_t *slot_of_expert);

/* moe_cache_free - wait for the device and release everything; NULL is a
 * no-op. */
void moe_cache_free(moe_expert_cache *c);

/*
 * Shortcut-connected MoE (dragon.c, "Shortcut-connected MoE": the MoE is
 * computed on sub-block-0's normed hidden state and its output is added at
 * the END of sub-block-1, "a designed overlap window"; §10: "thread the MoE
 * against sub-block-1's attention").  The MoE forward and sub-block-1's
 * attention run on two streams; the two calls below make that overlap work.
 *
 * moe_set_sm_budget - let the layer's persistent kernels (one CTA per SM)
 * use at most n_sms SMs, leaving the rest to work on other streams; n_sms
 * <= 0 restores all SMs.  Takes effect from the next forward.
 */
int moe_set_sm_budget(moe_ctx *ctx, int32_t n_sms);

/*
 * moe_decode_attention - softmax attention of one new token per sequence
 * against its key/value cache:
 *   out[b, h] = softmax(q[b, h] . K[b, :, c]^T / sqrt(d)) V[b, :, c],
 *   c = h / (n_heads / n_kv_heads).
 *   q        : device bf16 [B, n_heads, d];
 *   k_cache, v_cache : device bf16 [B, S, n_kv_heads, d];
 *   out      : device bf16 [B, n_heads, d];
 *   workspace: device, at least moe_attention_workspace_bytes(B, S,
 *              n_heads, d) bytes (f32 partial results; caller-owned).
 * d must be 128; n_heads / n_kv_heads one of 1, 2, 4, 8 (MOE_ERR_SHAPE
 * otherwise); pointers 16-byte aligned.  f32 arithmetic, bf16 output.  No
 * counterpart in the pages beyond its role: sub-block-1's attention, the
 * work the MoE overlaps.
 */
int64_t moe_attention_workspace_bytes(int64_t B, int64_t S, int32_t n_heads, int32_t head_dim);
int moe_decode_attention(const void *q, const void *k_cache, const void *v_cache, int64_t B,
                         int64_t S, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, void *out,
                         void *workspace, int64_t workspace_bytes, void *stream);

/*
 * moe_selftest_wait_timeout - exercise the bounded device-side waits.  Every
 * wait inside the layer's kernels (mbarriers of TMA copies and tensor-core
 * work, cross-CTA counters) gives up after a time limit and records
 * MOE_ERR_DEVICE_TIMEOUT instead of hanging the GPU.  This call enqueues one
 * CTA that holds tensor memory as those kernels do and waits, with the same
 * helpers, on an mbarrier that nothing arrives on and on a counter in the
 * context's workspace that nothing increments, `limit_ns` each; both waits
 * give up, the CTA frees its tensor memory and returns.
 *   limit_ns : 1 .. 1e9 nanoseconds per wait.
 *   which    : device int32 or NULL; receives the waits that gave up (bit 0
 *              the mbarrier, bit 1 the counter: 3 when both did).
 *   stream   : cudaStream_t or NULL.
 * Afterwards moe_status reports MOE_ERR_DEVICE_TIMEOUT once (and clears it);
 * the context stays usable.  No counterpart in the pages: it tests the
 * failure handling of this library.
 */
int moe_selftest_wait_timeout(moe_ctx *ctx, int64_t limit_ns, int32_t *which, void *stream);

/*
 * moe_route_noalloc - the routing step alone (steps 1 and 2 above) for callers
 * that may not allocate device memory once running: applications that hand
 * all device memory to their own allocator at start-up, or inference loops
 * with a fixed memory budget, where a cudaMalloc could fail or stall the
 * device.  It allocates nothing and needs no context: its temporary buffers
 * live in one statically sized device array of this library (about 269 KB,
 * held on every GPU that loads the library until the process exits).
 * There is no counterpart in the pages; it computes the same routing as
 * moe_layer_forward followed by moe_get_routing.
 *   hidden      : device, bf16 [T, H], 16-byte aligned; T <= 64.
 *   H           : multiple of 128, <= 65536.
 *   router_w    : device, f32 [E, H], 16-byte aligned; 1 <= E <= 1024.
 *   router_bias : device, f32 [E], or NULL.
 *   top_k       : 1..min(E, 32).
 *   idx, wts    : device outputs, int32 / f32 [T, k], rank order.
 *   counts      : device output, int32 [E].
 *   offsets     : device output, int32 [E+1].
 *   perm, inv   : device outputs, int32 [T*k].
 *   stream      : cudaStream_t or NULL.
 * Sizes beyond these limits return MOE_ERR_SHAPE; T = 0 is a no-op.  The
 * first call on a device looks up the array's device address (a host-side
 * query, done once per device, with that device current): make that first
 * call outside any stream capture.  Every call shares the one array and
 * clears the part that must start at zero; calls whose work overlaps on the
 * GPU (other streams, other host threads) race on it and must be serialised
 * by the caller.  Device-side errors (non-finite logits) are not reported.
 */
int moe_route_noalloc(const void *hidden, int64_t T, int64_t H, const float *router_w,
                      const float *router_bias, int64_t E, int32_t top_k, int32_t *idx, float *wts,
                      int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8MOE_H */
