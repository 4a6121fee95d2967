// Hooks of the context's forward for other parts of the library (not part
// of the C ABI): the routing and expert phases of one forward, run
// separately, and the active-expert list of the last routing.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8moe.h"

namespace fp8moe {

// Checks a forward's arguments as moe_layer_forward does; *path receives the
// expert path a forward of T tokens takes.
int ctx_check_forward(moe_ctx *c, const void *hidden, int64_t T, const float *rw, const float *rb,
                      const uint8_t *w13, const float *s13, const uint8_t *w2, const float *s2,
                      int32_t k, const void *out, int *path);
// Routing (everything before the expert kernels), enqueued on s.
int ctx_route(moe_ctx *c, const __nv_bfloat16 *x, int64_t T, const float *rw, const float *rb,
              int k, int path, cudaStream_t s);
// Expert kernels and combine on the context's routing, enqueued on s.  With
// slot_of (device int32 [E]), w13 / w2 hold n_slabs expert slabs and expert
// e's codes are slab slot_of[e]; s13 / s2 stay indexed by expert.
int ctx_experts(moe_ctx *c, const __nv_bfloat16 *x, int64_t T, const uint8_t *w13,
                const float *s13, const uint8_t *w2, const float *s2, int k, int path,
                __nv_bfloat16 *out, cudaStream_t s, const int32_t *slot_of = nullptr,
                int64_t n_slabs = 0);
// Copies the number of active experts and their list (ascending) into the
// host buffer buf[0], buf[1 ..] (pinned, n_experts + 1 ints) and waits for s.
int ctx_active_experts(moe_ctx *c, int32_t *buf, cudaStream_t s);
const moe_config *ctx_config(const moe_ctx *c);

}  // namespace fp8moe
