// Check of the bounded-wait machinery every tensor-core kernel relies on.
//
// One CTA initialises an mbarrier that nothing ever arrives on and waits for it with the
// same bounded wait the kernels use (mbar_wait_bounded, %globaltimer), under a caller-given
// limit.  The wait must give up, write MOE_ERR_TIMEOUT into the workspace status word and
// let the CTA exit: the context stays usable and the next call runs normally.  No fault,
// no trap, nothing left in flight (the barrier lives in the CTA's shared memory).
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__global__ void __launch_bounds__(32, 1) wait_bound_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    // phase 0 never completes: nothing arrives
    mbar_wait_bounded(smem_u32(&bar), 0u, &abort_flag, status, limit_ns);
  }
  __syncwarp();
}

}  // namespace

cudaError_t launch_wait_bound_check(int32_t* status, uint64_t limit_ns, cudaStream_t s) {
  wait_bound_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
