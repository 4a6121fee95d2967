// Self-test of the bounded device-side waits that every kernel of the layer
// relies on instead of waiting forever.
//
// One CTA allocates tensor memory as the layer's tensor-core kernels do, then
// waits with the same helpers they use (sm100_ptx.cuh) on an mbarrier that
// nothing arrives on and on a global counter that nothing increments, each
// with a short limit.  Both waits give up; the kernel records the timeout in
// the context's error flag (read by moe_status), reports which waits gave up,
// frees its tensor memory on the way out and returns, so the context stays
// usable.  Nothing here faults or traps: the failure is only the wait that
// runs out.
#include "common.cuh"
#include "kernels.h"
#include "sm100_ptx.cuh"

namespace fp8moe {
using namespace sm100;

namespace {

constexpr uint32_t kSelftestTmemCols = 32;

__global__ void __launch_bounds__(64, 1) bounded_wait_selftest_kernel(const int32_t *idle_counter,
                                                                      uint64_t limit_ns, int *err,
                                                                      int32_t *which) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base, kSelftestTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    int bits = 0;
    // phase 0 of the barrier never completes: no thread arrives on it
    if (!mbar_wait(&bar, 0u, &abort_flag, limit_ns)) bits |= 1;
    // the counter stays at 0
    if (!wait_counter_ge(idle_counter, 1, &abort_flag, limit_ns)) bits |= 2;
    if (which != nullptr) *which = bits;
    if (bits != 0) {
      abort_flag = 1;
      set_error(err, DEV_ERR_TIMEOUT);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kSelftestTmemCols);
  }
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(const int32_t *idle_counter, uint64_t limit_ns, int *err,
                                         int32_t *which, cudaStream_t s) {
  bounded_wait_selftest_kernel<<<1, 64, 0, s>>>(idle_counter, limit_ns, err, which);
  return cudaGetLastError();
}

}  // namespace fp8moe
