// E4M3 encoding shared by the row quantiser (fp8.cu) and the W8A8 expert
// kernel's activation quantisation: round to nearest even, magnitudes past 448
// saturated to 448 (the conversion instructions' satfinite mode).
#pragma once
#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {

// Four values to four E4M3 codes, the first in the low byte.
__device__ __forceinline__ uint32_t e4m3_pack4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xFFFFu) | (hi << 16);
}

// A row's scale from its largest magnitude: max / 448 (IEEE division), 1 for a zero row.
__device__ __forceinline__ float e4m3_row_scale(float amax) { return amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f; }

}  // namespace moe
