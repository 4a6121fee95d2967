// Routing (logits, top-k selection, pair sort) without any device allocation.
//
// Some callers cannot call cudaMalloc once they are running: applications
// that reserve all device memory for their own allocator at start-up, or
// inference loops with a fixed memory budget, where an allocation could fail
// under memory pressure or stall the device.  moe_route_noalloc serves them:
// the caller passes inputs and outputs, and every temporary buffer the
// routing kernel needs lives in the file-scope array below, which each GPU
// that loads this library holds until the process exits.
#include <cuda.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "fp8moe.h"
#include "kernels.h"

namespace {

constexpr int64_t kMaxT = 64;     // largest batch the array is sized for
constexpr int64_t kMaxE = 1024;   // largest expert count

// layout, in 4-byte words
constexpr size_t kLogits = 0;                         // f32 [kMaxT * kMaxE]
constexpr size_t kWnorm = kLogits + kMaxT * kMaxE;    // f32 [kMaxE]
constexpr size_t kXnorm = kWnorm + kMaxE;             // f32 [kMaxT]
constexpr size_t kTicket = kXnorm + kMaxT;            // i32, 0 between calls
constexpr size_t kErr = kTicket + 1;                  // i32 device error bits of this call (not reported)
constexpr size_t kActive = kTicket + 4;               // i32 [kMaxE]
constexpr size_t kNActive = kActive + kMaxE;          // i32
constexpr size_t kTiles = kNActive + 4;               // i32 [kMaxE + 1]
constexpr size_t kWords = kTiles + kMaxE + 4;

static __device__ __align__(256) uint32_t g_route_scratch[kWords];  // ~269 KB

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Resolved {
  CUcontext ctx;  // context the address was looked up in
  uint32_t *ptr;  // device address of the array in that context
};
Resolved g_scratch[kMaxDevices] = {};

// The driver's current context (nullptr when none, or when the query is
// unavailable).
CUcontext current_context() {
  using Fn = CUresult (*)(CUcontext *);
  static Fn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<Fn>(nullptr);
    return reinterpret_cast<Fn>(p);
  }();
  CUcontext c = nullptr;
  if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of the array on the current device.  The array's host-side
// name is not a device address; the address is looked up with that device
// current and kept for as long as the same context is current, so that a
// reset of the device (a new context, where the module and its array may sit
// elsewhere) leads to a fresh lookup.
int scratch_on_current_device(uint32_t **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  const CUcontext ctx = current_context();
  if (g_scratch[dev].ptr == nullptr || ctx == nullptr || g_scratch[dev].ctx != ctx) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    g_scratch[dev].ptr = static_cast<uint32_t *>(p);
    g_scratch[dev].ctx = current_context();  // the lookup made the runtime's context current
  }
  *out = g_scratch[dev].ptr;
  return MOE_OK;
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

extern "C" int moe_route_noalloc(const void *hidden, int64_t T, int64_t H, const float *router_w,
                                 const float *router_bias, int64_t E, int32_t top_k, int32_t *idx,
                                 float *wts, int32_t *counts, int32_t *offsets, int32_t *perm,
                                 int32_t *inv, void *stream) {
  if (T < 0) return MOE_ERR_ARG;
  if (T > kMaxT || E < 1 || E > kMaxE || H <= 0 || H % 128 != 0 || H > 65536 || top_k < 1 ||
      top_k > 32 || top_k > E)
    return MOE_ERR_SHAPE;
  if (T == 0) return MOE_OK;
  if (!hidden || !router_w || !idx || !wts || !counts || !offsets || !perm || !inv)
    return MOE_ERR_ARG;
  if (!aligned(hidden, 16) || !aligned(router_w, 16) || (router_bias && !aligned(router_bias, 4)) ||
      !aligned(idx, 4) || !aligned(wts, 4) || !aligned(counts, 4) || !aligned(offsets, 4) ||
      !aligned(perm, 4) || !aligned(inv, 4))
    return MOE_ERR_ALIGN;
  uint32_t *sc = nullptr;
  int rc = scratch_on_current_device(&sc);
  if (rc != MOE_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float *logits = reinterpret_cast<float *>(sc + kLogits);
  float *wnorm = reinterpret_cast<float *>(sc + kWnorm);
  float *xnorm = reinterpret_cast<float *>(sc + kXnorm);
  int32_t *ticket = reinterpret_cast<int32_t *>(sc + kTicket);
  int32_t *active = reinterpret_cast<int32_t *>(sc + kActive);
  int32_t *n_active = reinterpret_cast<int32_t *>(sc + kNActive);
  int32_t *tiles = reinterpret_cast<int32_t *>(sc + kTiles);
  int *err = reinterpret_cast<int *>(sc + kErr);
  // the completion ticket must start at zero (the previous call leaves it at
  // zero unless it was interrupted), and this call's error bits start clear:
  // the two words are adjacent
  static_assert(kErr == kTicket + 1, "ticket and error word are cleared together");
  if (cudaMemsetAsync(ticket, 0, 2 * sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  const cudaError_t e = fp8moe::launch_route_decode(
      static_cast<const __nv_bfloat16 *>(hidden), T, router_w, router_bias, E, H, top_k,
      fp8moe::router_gamma(H), logits, wnorm, xnorm, nullptr, nullptr, ticket, idx, wts,
      counts, offsets, perm, inv, active, n_active, tiles, fp8moe::kTileM, nullptr, err, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
