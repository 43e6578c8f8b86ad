// FP8 (E4M3) expert weights with one fp32 scale per output row: the
// quantiser the FP8 expert path is fed from.
//
// "Hy3 Preview inference optimisation case" lists W8A8 quantised deployments
// and quantisation inside the FusedMoE chain without fixing a format.  Here:
// OCP E4M3 codes (largest finite magnitude 448), scale = max|row| / 448 in fp32
// (1 for an all-zero row), code = E4M3 nearest-even of w / scale (the fp32
// quotient rounded to nearest even), saturated at 448.  The expert kernel feeds the code values to the
// MMAs and multiplies each row's fp32 accumulator by the row's scale.
#include "fp8.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {
constexpr int kQThreads = 256;  // eight rows (one per warp) per CTA step
}  // namespace

// One warp per row: the row maximum first, then the codes, 8 values per lane
// step (16-byte loads of bf16, 8-byte stores of codes).
__global__ void __launch_bounds__(kQThreads) quantize_rows_kernel(const __nv_bfloat16 *__restrict__ src,
                                                                  uint8_t *__restrict__ q, float *__restrict__ scale,
                                                                  long long rows, int cols) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int n8 = cols >> 3;
  for (long long r = (long long)blockIdx.x * (kQThreads / 32) + (threadIdx.x >> 5); r < rows;
       r += (long long)gridDim.x * (kQThreads / 32)) {
    const uint4 *row = reinterpret_cast<const uint4 *>(src + r * cols);
    float amax = 0.0f;
    for (int i = lane; i < n8; i += 32) {
      const uint4 v = row[i];
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(u[j] << 16)), fabsf(__uint_as_float(u[j] & 0xFFFF0000u))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = e4m3_row_scale(amax), rs = __frcp_rn(s);
    if (lane == 0) scale[r] = s;
    uint2 *out = reinterpret_cast<uint2 *>(q + r * cols);
    for (int i = lane; i < n8; i += 32) {
      const uint4 v = row[i];
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
      float f[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        f[2 * j] = e4m3_quotient(__uint_as_float(u[j] << 16), s, rs);
        f[2 * j + 1] = e4m3_quotient(__uint_as_float(u[j] & 0xFFFF0000u), s, rs);
      }
      out[i] = make_uint2(e4m3_pack4(f[0], f[1], f[2], f[3]), e4m3_pack4(f[4], f[5], f[6], f[7]));
    }
  }
}

cudaError_t launch_quantize_rows(const __nv_bfloat16 *src, uint8_t *q, float *scale, long long rows, int cols,
                                 cudaStream_t stream) {
  int dev = 0, nsm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (rows + kQThreads / 32 - 1) / (kQThreads / 32);
  const long long cap = (long long)(nsm > 0 ? nsm : 1) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  void *args[] = {(void *)&src, (void *)&q, (void *)&scale, (void *)&rows, (void *)&cols};
  return launch_ex((const void *)quantize_rows_kernel, dim3((unsigned)blocks), dim3(kQThreads), 0, stream, true, 1,
                   args);
}

}  // namespace moe
