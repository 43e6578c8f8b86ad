// SiLU(gate) * up for the gate/up epilogue (step a6: a = g / (1 + e^-g) * u),
// shared by the expert kernel and its self-test entry point.
#pragma once
#include <stdint.h>

namespace moe {

// One special-function operation per element (the epilogue of a wide tile is
// bound by them):
//   e = 2^(-g log2 e) by the hardware base-2 exponential (ex2.approx), its
//       argument capped at 120 so that 1 + e stays a normal float;
//   1 / (1 + e) by Newton-Raphson iteration for the reciprocal,
//       r <- r (2 - d r), twice, from a linear initial estimate on the float's
//       bit pattern, r0 = bits^-1(K - bits(d)) (the integer-subtraction seed of
//       the "fast inverse" family of methods).  K = 0x7EF311C0 was found in this
//       project by a search that minimises the seed's worst relative error over
//       one binade (5.05 %); two steps bring it to 6.6e-6.
// Accuracy (checked on the device against float64 by moe_selftest_silu):
// relative error within 1e-5 of SiLU(g) * u for g >= -83; for g < -83 the cap
// leaves |result| <= |g u| 2^-119 (the true value is below 1e-34 there), far
// below the bf16 rounding that follows.  SiLU(0) * u = 0 exactly.
__device__ __forceinline__ float silu_mul(float g, float u) {
  const float x = fminf(-1.4426950409f * g, 120.0f);
  float e;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x));
  const float d = 1.0f + e;
  float r = __int_as_float(0x7EF311C0 - __float_as_int(d));
  r = r * fmaf(-d, r, 2.0f);
  r = r * fmaf(-d, r, 2.0f);
  return g * u * r;
}

}  // namespace moe
