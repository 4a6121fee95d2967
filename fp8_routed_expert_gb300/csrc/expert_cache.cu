// Experts larger than device memory: the expert weights stay in host memory
// and a fixed number of expert slots in HBM hold the ones in use, streamed in
// over NVLink-C2C (DeepSeek-V4.1-Flash post, "Bytes per token decide
// everything" and v4 of "Making it faster": a cache in front of the slow
// tier, copies of the experts a token needs, and the next layer's experts
// guessed from its router and prefetched into the gap; Qwen post, "Where the
// time actually goes": speculative copies started one layer early).
//
// GB300 design.  The cache is two device buffers of n_slots expert slabs
// (W13 codes [n_slots, 2I, H], W2 codes [n_slots, H, I]) and a table
// slot_of[E]; the layer's own kernels read expert e's codes from slab
// slot_of[e] (its block scales stay resident, indexed by e).  A forward
// routes first, reads the active-expert list back (the per-layer host sync
// the pages measure as cheap), copies the missing experts into least
// recently used slabs on the forward's stream, uploads the table and runs
// the expert kernels.  Prefetches copy on a second stream into slabs that no
// forward in flight uses; the next forward waits for them with an event.
#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "ctx_internal.h"
#include "fp8moe.h"

using namespace fp8moe;

namespace {

// One matrix set (W13 or W2) of all experts: the host copy and the device
// slabs of the cache.
struct Matrix {
  const uint8_t *host = nullptr;
  size_t bytes = 0;  // per expert
  bool registered = false;
  uint8_t *slabs = nullptr;  // device [n_slots][bytes]
};

}  // namespace

struct moe_expert_cache {
  moe_ctx *ctx = nullptr;
  int device = 0;
  int64_t E = 0, n_slots = 0;
  Matrix m[2];                    // W13, W2
  std::vector<int> slot_expert;   // expert held by each slot, -1 if none
  std::vector<int> expert_slot;   // slot of each expert, -1 if not cached
  std::vector<uint64_t> last_use; // per slot: tick of the last forward or prefetch that used it
  std::vector<char> in_use;       // per slot: needed by the last forward (may still run)
  std::vector<char> prefetched;   // per slot: filled by a prefetch and not yet used by a forward
  uint64_t tick = 0;
  int32_t *act = nullptr;         // pinned host: n_active, active list
  int32_t *slot_host = nullptr;   // pinned host: slot of every expert (-1: none)
  int32_t *slot_dev = nullptr;    // device copy read by the expert kernels
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t prefetch_done = nullptr;
  bool prefetch_pending = false;
  int64_t stats[MOE_CACHE_STATS] = {};
  // next-layer guesses (device buffers of moe_route_noalloc, pinned readback)
  int32_t *g_idx = nullptr, *g_counts = nullptr, *g_offsets = nullptr, *g_perm = nullptr,
          *g_inv = nullptr;
  float *g_wts = nullptr;
  int32_t *g_idx_host = nullptr;
  cudaStream_t guess_stream = nullptr;
};

namespace {

constexpr int64_t kGuessMaxT = 64, kGuessMaxK = 32;

void destroy(moe_expert_cache *c) {
  if (c->copy_stream) cudaStreamSynchronize(c->copy_stream);
  for (int i = 0; i < 2; ++i) {
    Matrix &mx = c->m[i];
    if (mx.slabs) cudaFree(mx.slabs);
    if (mx.registered) cudaHostUnregister(const_cast<uint8_t *>(mx.host));
  }
  if (c->act) cudaFreeHost(c->act);
  if (c->slot_host) cudaFreeHost(c->slot_host);
  if (c->slot_dev) cudaFree(c->slot_dev);
  if (c->g_idx_host) cudaFreeHost(c->g_idx_host);
  for (void *p : {(void *)c->g_idx, (void *)c->g_counts, (void *)c->g_offsets, (void *)c->g_perm,
                  (void *)c->g_inv, (void *)c->g_wts})
    if (p) cudaFree(p);
  if (c->prefetch_done) cudaEventDestroy(c->prefetch_done);
  if (c->copy_stream) cudaStreamDestroy(c->copy_stream);
  if (c->guess_stream) cudaStreamDestroy(c->guess_stream);
  delete c;
}

// Least recently used slot that may be refilled now: not needed by the last
// forward, not filled earlier in this same prefetch batch (`batch` marks),
// preferring free slots.  -1 if none.
int64_t victim(const moe_expert_cache *c, const std::vector<char> &batch) {
  int64_t best = -1;
  for (int64_t s = 0; s < c->n_slots; ++s) {
    if (c->in_use[s] || batch[s]) continue;
    if (c->slot_expert[s] < 0) return s;
    if (best < 0 || c->last_use[s] < c->last_use[best]) best = s;
  }
  return best;
}

// Puts expert e into slot s (the expert it held leaves the cache) and
// enqueues the copies of e's W13 and W2 codes from host memory on `st`.
int load_into(moe_expert_cache *c, int e, int64_t s, cudaStream_t st) {
  const int old = c->slot_expert[s];
  if (old >= 0) {
    c->expert_slot[old] = -1;
    c->slot_host[old] = -1;
    c->stats[MOE_CACHE_EVICTIONS] += 1;
  }
  for (int i = 0; i < 2; ++i) {
    Matrix &mx = c->m[i];
    if (cudaMemcpyAsync(mx.slabs + (size_t)s * mx.bytes, mx.host + (size_t)e * mx.bytes, mx.bytes,
                        cudaMemcpyHostToDevice, st) != cudaSuccess)
      return MOE_ERR_CUDA;
    c->stats[MOE_CACHE_BYTES_COPIED] += (int64_t)mx.bytes;
  }
  c->slot_expert[s] = e;
  c->expert_slot[e] = (int)s;
  c->slot_host[e] = (int32_t)s;
  return MOE_OK;
}

// Waits for the copies of the last prefetch batch (their slots may then be
// refilled).
int settle_prefetch(moe_expert_cache *c) {
  if (!c->prefetch_pending) return MOE_OK;
  if (cudaEventSynchronize(c->prefetch_done) != cudaSuccess) return MOE_ERR_CUDA;
  c->prefetch_pending = false;
  return MOE_OK;
}

}  // namespace

extern "C" {

int moe_cache_init(moe_expert_cache **out, moe_ctx *ctx, const uint8_t *w13_host,
                   const uint8_t *w2_host, int64_t n_slots) {
  if (out == nullptr) return MOE_ERR_ARG;
  *out = nullptr;
  if (ctx == nullptr || w13_host == nullptr || w2_host == nullptr) return MOE_ERR_ARG;
  const moe_config *cfg = ctx_config(ctx);
  const int64_t E = cfg->n_experts, H = cfg->hidden, I = cfg->inter;
  if (n_slots < 1 || n_slots > E) return MOE_ERR_SHAPE;
  if (cudaSetDevice(cfg->device) != cudaSuccess) return MOE_ERR_CUDA;
  const size_t b13 = (size_t)(2 * I * H), b2 = (size_t)(H * I);

  moe_expert_cache *c = new (std::nothrow) moe_expert_cache();
  if (c == nullptr) return MOE_ERR_NOMEM;
  c->ctx = ctx;
  c->device = cfg->device;
  c->E = E;
  c->n_slots = n_slots;
  c->m[0].host = w13_host;
  c->m[0].bytes = b13;
  c->m[1].host = w2_host;
  c->m[1].bytes = b2;
  c->slot_expert.assign(n_slots, -1);
  c->expert_slot.assign(E, -1);
  c->last_use.assign(n_slots, 0);
  c->in_use.assign(n_slots, 0);
  c->prefetched.assign(n_slots, 0);
  int rc = MOE_OK;
  for (int i = 0; i < 2 && rc == MOE_OK; ++i) {
    Matrix &mx = c->m[i];
    const size_t total = (size_t)E * mx.bytes;
    // page-locked host memory lets the copies run asynchronously at full
    // link speed; memory that already is page-locked (cudaHostAlloc or an
    // earlier registration) is used as it is
    cudaPointerAttributes pa;
    const bool locked = cudaPointerGetAttributes(&pa, mx.host) == cudaSuccess &&
                        pa.type == cudaMemoryTypeHost;
    cudaGetLastError();
    if (!locked) {
      const cudaError_t er =
          cudaHostRegister(const_cast<uint8_t *>(mx.host), total, cudaHostRegisterDefault);
      if (er == cudaSuccess) mx.registered = true;
      else if (er == cudaErrorHostMemoryAlreadyRegistered) cudaGetLastError();
      else { cudaGetLastError(); rc = MOE_ERR_CUDA; break; }
    }
    if (cudaMalloc(&mx.slabs, (size_t)n_slots * mx.bytes) != cudaSuccess) {
      cudaGetLastError();
      mx.slabs = nullptr;
      rc = MOE_ERR_NOMEM;
      break;
    }
  }
  const size_t gbytes = (size_t)kGuessMaxT * kGuessMaxK * 4;
  if (rc == MOE_OK &&
      (cudaMallocHost(&c->act, (size_t)(E + 1) * sizeof(int32_t)) != cudaSuccess ||
       cudaMallocHost(&c->slot_host, (size_t)E * sizeof(int32_t)) != cudaSuccess ||
       cudaMalloc(&c->slot_dev, (size_t)E * sizeof(int32_t)) != cudaSuccess ||
       cudaMallocHost(&c->g_idx_host, gbytes) != cudaSuccess ||
       cudaMalloc(&c->g_idx, gbytes) != cudaSuccess || cudaMalloc(&c->g_wts, gbytes) != cudaSuccess ||
       cudaMalloc(&c->g_perm, gbytes) != cudaSuccess || cudaMalloc(&c->g_inv, gbytes) != cudaSuccess ||
       cudaMalloc(&c->g_counts, (size_t)E * 4) != cudaSuccess ||
       cudaMalloc(&c->g_offsets, (size_t)(E + 1) * 4) != cudaSuccess ||
       cudaStreamCreateWithFlags(&c->copy_stream, cudaStreamNonBlocking) != cudaSuccess ||
       cudaStreamCreateWithFlags(&c->guess_stream, cudaStreamNonBlocking) != cudaSuccess ||
       cudaEventCreateWithFlags(&c->prefetch_done, cudaEventDisableTiming) != cudaSuccess)) {
    cudaGetLastError();
    rc = MOE_ERR_NOMEM;
  }
  if (rc != MOE_OK) {
    destroy(c);
    return rc;
  }
  for (int64_t e = 0; e < E; ++e) c->slot_host[e] = -1;
  *out = c;
  return MOE_OK;
}

void moe_cache_free(moe_expert_cache *c) {
  if (c == nullptr) return;
  cudaSetDevice(c->device);
  cudaDeviceSynchronize();  // no kernel may still read the slabs freed below
  destroy(c);
}

int moe_cache_forward(moe_expert_cache *c, const void *hidden, int64_t T, const float *router_w,
                      const float *router_bias, const float *s13, const float *s2, int32_t top_k,
                      void *out, void *stream) {
  if (c == nullptr) return MOE_ERR_ARG;
  int path = 0;
  // the slab buffers stand in for the weight pointers in the checks
  int rc = ctx_check_forward(c->ctx, hidden, T, router_w, router_bias, c->m[0].slabs, s13,
                             c->m[1].slabs, s2, top_k, out, &path);
  if (rc != MOE_OK || T == 0) return rc;
  if (cudaSetDevice(c->device) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16 *x = static_cast<const __nv_bfloat16 *>(hidden);
  if ((rc = ctx_route(c->ctx, x, T, router_w, router_bias, top_k, path, s)) != MOE_OK) return rc;
  // the active experts; the wait also retires the previous forward's kernels
  if ((rc = ctx_active_experts(c->ctx, c->act, s)) != MOE_OK) return rc;
  const int64_t n_act = c->act[0];
  if (n_act < 0 || n_act > c->E) return MOE_ERR_DEVICE;
  if (n_act > c->n_slots) return MOE_ERR_NOMEM;  // this batch's experts do not fit the slots
  std::fill(c->in_use.begin(), c->in_use.end(), 0);
  c->tick += 1;
  // hits first, so that they are not chosen as victims for the misses
  for (int64_t i = 0; i < n_act; ++i) {
    const int e = c->act[1 + i];
    if (e < 0 || e >= c->E) return MOE_ERR_DEVICE;
    const int sl = c->expert_slot[e];
    if (sl >= 0) {
      c->in_use[sl] = 1;
      c->last_use[sl] = c->tick;
      c->stats[MOE_CACHE_HITS] += 1;
      if (c->prefetched[sl]) {
        c->stats[MOE_CACHE_PREFETCH_USED] += 1;
        c->prefetched[sl] = 0;
      }
    }
  }
  std::vector<char> none(c->n_slots, 0);
  for (int64_t i = 0; i < n_act; ++i) {
    const int e = c->act[1 + i];
    if (c->expert_slot[e] >= 0) continue;
    if ((rc = settle_prefetch(c)) != MOE_OK) return rc;  // no slot is refilled under a copy in flight
    const int64_t sl = victim(c, none);
    if (sl < 0) return MOE_ERR_NOMEM;
    if ((rc = load_into(c, e, sl, s)) != MOE_OK) return rc;
    c->in_use[sl] = 1;
    c->prefetched[sl] = 0;
    c->last_use[sl] = c->tick;
    c->stats[MOE_CACHE_MISSES] += 1;
  }
  // experts prefetched on the copy stream may still be arriving
  if (c->prefetch_pending && cudaStreamWaitEvent(s, c->prefetch_done, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  // the table reaches the device in stream order; a prefetch that changes
  // slot_host before this copy runs only changes entries of experts that
  // this forward does not use (its slots are in use and never refilled)
  if (cudaMemcpyAsync(c->slot_dev, c->slot_host, (size_t)c->E * sizeof(int32_t),
                      cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return ctx_experts(c->ctx, x, T, c->m[0].slabs, s13, c->m[1].slabs, s2, top_k, path,
                     static_cast<__nv_bfloat16 *>(out), s, c->slot_dev, c->n_slots);
}

int moe_cache_prefetch(moe_expert_cache *c, const int32_t *experts, int64_t n) {
  if (c == nullptr || (n > 0 && experts == nullptr) || n < 0) return MOE_ERR_ARG;
  if (cudaSetDevice(c->device) != cudaSuccess) return MOE_ERR_CUDA;
  int rc = settle_prefetch(c);
  if (rc != MOE_OK) return rc;
  std::vector<char> batch(c->n_slots, 0);
  int64_t issued = 0;
  for (int64_t i = 0; i < n; ++i) {
    const int e = experts[i];
    if (e < 0 || e >= c->E) return MOE_ERR_ARG;
    if (c->expert_slot[e] >= 0) continue;
    const int64_t sl = victim(c, batch);
    if (sl < 0) break;  // every slot is needed by the forward in flight or this batch
    if ((rc = load_into(c, e, sl, c->copy_stream)) != MOE_OK) return rc;
    batch[sl] = 1;
    c->prefetched[sl] = 1;
    c->last_use[sl] = c->tick;
    c->stats[MOE_CACHE_PREFETCHED] += 1;
    ++issued;
  }
  if (issued > 0) {
    if (cudaEventRecord(c->prefetch_done, c->copy_stream) != cudaSuccess) return MOE_ERR_CUDA;
    c->prefetch_pending = true;
  }
  return (int)issued;
}

int moe_cache_guess(moe_expert_cache *c, const void *hidden, int64_t T, const float *router_w,
                    const float *router_bias, int32_t top_k, int32_t n_guess, int32_t *experts_out) {
  if (c == nullptr || hidden == nullptr || router_w == nullptr || experts_out == nullptr ||
      n_guess < 0)
    return MOE_ERR_ARG;
  const int64_t E = c->E, H = ctx_config(c->ctx)->hidden;
  if (T < 1 || T > kGuessMaxT || top_k < 1 || top_k > kGuessMaxK || top_k > E) return MOE_ERR_SHAPE;
  if (cudaSetDevice(c->device) != cudaSuccess) return MOE_ERR_CUDA;
  int rc = moe_route_noalloc(hidden, T, H, router_w, router_bias, E, top_k, c->g_idx, c->g_wts,
                             c->g_counts, c->g_offsets, c->g_perm, c->g_inv, c->guess_stream);
  if (rc != MOE_OK) return rc;
  if (cudaMemcpyAsync(c->g_idx_host, c->g_idx, (size_t)(T * top_k) * 4, cudaMemcpyDeviceToHost,
                      c->guess_stream) != cudaSuccess ||
      cudaStreamSynchronize(c->guess_stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  // rank: tokens choosing the expert (more first), then its best rank, then id
  std::vector<int64_t> votes(E, 0), best(E, top_k);
  for (int64_t t = 0; t < T; ++t)
    for (int r = 0; r < top_k; ++r) {
      const int e = c->g_idx_host[t * top_k + r];
      if (e < 0 || e >= E) return MOE_ERR_DEVICE;
      votes[e] += 1;
      best[e] = std::min<int64_t>(best[e], r);
    }
  std::vector<int> order;
  for (int e = 0; e < E; ++e)
    if (votes[e] > 0) order.push_back(e);
  std::sort(order.begin(), order.end(), [&](int a, int b) {
    if (votes[a] != votes[b]) return votes[a] > votes[b];
    if (best[a] != best[b]) return best[a] < best[b];
    return a < b;
  });
  const int64_t m = std::min<int64_t>(n_guess, (int64_t)order.size());
  for (int64_t i = 0; i < m; ++i) experts_out[i] = order[i];
  return (int)m;
}

int moe_cache_stats(const moe_expert_cache *c, int64_t *out, int32_t n) {
  if (c == nullptr || out == nullptr || n < 0) return MOE_ERR_ARG;
  for (int i = 0; i < n && i < MOE_CACHE_STATS; ++i) out[i] = c->stats[i];
  return MOE_OK;
}

int moe_cache_resident(const moe_expert_cache *c, int32_t *slot_of_expert) {
  if (c == nullptr || slot_of_expert == nullptr) return MOE_ERR_ARG;
  for (int64_t e = 0; e < c->E; ++e) slot_of_expert[e] = c->expert_slot[e];
  return MOE_OK;
}

}  // extern "C"
