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

// x / s rounded to nearest even, given rs = 1/s rounded to nearest even (one
// reciprocal per row instead of one division per value).  The product q0 = x rs
// is within one ulp of x / s, so the remainder x - q0 s is exact in one fused
// multiply-add, and q0 + remainder * rs rounds to the correctly rounded quotient
// (Markstein's theorem; P. Markstein, "Computation of elementary functions on
// the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990).  It needs
// no overflow or gradual underflow, which holds here: |x / s| <= 448 and
// quotients below fp32's normal range quantise to zero whatever their last bit.
// The theorem says nothing of signed zeros (the correction turns -0 into +0):
// the quotient takes the sign of q0, which is that of x.
__device__ __forceinline__ float e4m3_quotient(float x, float s, float rs) {
  const float q0 = x * rs;
  return copysignf(fmaf(fmaf(-q0, s, x), rs, q0), q0);
}

}  // namespace moe
