// Self-test of the bounded waits every kernel of this library uses: one CTA
// waits on an mbarrier phase that nothing completes, with a short limit, and
// must give up, record MOE_DEVERR_TIMEOUT in the workspace error word and
// return -- the GPU context stays usable.  No fault, trap or endless loop.
#include "internal.h"
#include "ptx.cuh"

namespace moe {

__global__ void wait_timeout_kernel(unsigned *err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // one arrival expected; none ever comes
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_for(smem_u32(&bar), 0, err, &abort_flag, limit_ns);
}

cudaError_t launch_wait_timeout(unsigned *err, unsigned long long limit_ns, cudaStream_t stream) {
  void *args[] = {(void *)&err, (void *)&limit_ns};
  return launch_ex((const void *)wait_timeout_kernel, dim3(1), dim3(32), 0, stream, false, 1, args);
}

}  // namespace moe
