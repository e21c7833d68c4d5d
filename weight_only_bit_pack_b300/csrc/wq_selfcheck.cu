// Self-check of the device error channel: one thread waits, with the same
// bounded wait the operator kernels use, for an mbarrier phase that nothing
// completes. When the budget runs out the wait records WQ_ERR_DEVICE_TIMEOUT
// and the place in the workspace status word and the kernel returns, which is
// the path an operator kernel takes when a wait for other thread blocks gives
// up. No fault, trap or endless loop is involved.
#include "wq_internal.h"
#include "wq_sm100.cuh"
#include "wq_sync.cuh"

namespace wq {
namespace {

__global__ void timeout_check_kernel(uint32_t *status, long long budget) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  sm100::mbar_init(sm100::smem_u32(&bar), 1);  // one arrival, which never comes
  abort_flag = 0;
  sm100::fence_mbar_init();
  wait_bar(sm100::smem_u32(&bar), 0u, &abort_flag, status, WQ_WHERE_SELF_CHECK, budget);
}

}  // namespace

cudaError_t launch_timeout_check(uint32_t *status, long long budget, cudaStream_t s) {
  timeout_check_kernel<<<1, 32, 0, s>>>(status, budget);
  return cudaGetLastError();
}

}  // namespace wq
