// Self-tests of device building blocks:
//  - the bounded waits every kernel of this library uses: one CTA waits on an
//    mbarrier phase that nothing completes, with a short limit, and must give
//    up, record MOE_DEVERR_TIMEOUT in the workspace error word and return -- the
//    GPU context stays usable.  No fault, trap or endless loop.
//  - the epilogue's SiLU(gate) * up, evaluated element-wise on given inputs so
//    that its error can be measured against float64 on the host.
#include "internal.h"
#include "ptx.cuh"
#include "silu.cuh"

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

__global__ void __launch_bounds__(256) silu_selftest_kernel(const float *__restrict__ g, const float *__restrict__ u,
                                                            float *__restrict__ out, long long n) {
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < n; i += 256ll * gridDim.x) out[i] = silu_mul(g[i], u[i]);
}

cudaError_t launch_silu_selftest(const float *g, const float *u, float *out, long long n, cudaStream_t stream) {
  const long long blocks = (n + 255) / 256;
  void *args[] = {(void *)&g, (void *)&u, (void *)&out, (void *)&n};
  return launch_ex((const void *)silu_selftest_kernel, dim3((unsigned)(blocks < 1024 ? blocks : 1024)), dim3(256), 0,
                   stream, false, 1, args);
}

}  // namespace moe
