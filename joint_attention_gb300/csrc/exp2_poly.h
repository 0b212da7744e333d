// exp2_poly.h — 2^x on the FMA pipe, for part of the softmax exponentials.
//
// Method (derived in gen_exp2_poly.py, next to this file): round-to-nearest
// range reduction x = n + f, f in [-1/2, 1/2], then 2^f from the degree-3
// polynomial that minimises the maximum relative error on that interval
// (Remez exchange), and 2^n added to the result's exponent field.  Maximum
// relative error 7.5e-5 (float32 Horner), far below the 2^-9 rounding of the
// bf16 probabilities it feeds.  Valid for x >= -125 (smaller x is clamped:
// the result is then ~2e-38 instead of 0); NaN/inf inputs are not expected.
#pragma once

namespace jattn {

constexpr float kExp2C0 = 0.9999280571937561f;
constexpr float kExp2C1 = 0.6932609677314758f;
constexpr float kExp2C2 = 0.2426111251115799f;
constexpr float kExp2C3 = 0.0551716685295105f;

__device__ __forceinline__ float exp2_poly(float x) {
  x = fmaxf(x, -125.0f);
  // Adding 1.5 * 2^23 leaves round(x) in the low mantissa bits of t.
  const float t = x + 12582912.0f;
  const float n = t - 12582912.0f;
  const float f = x - n;
  float p = fmaf(kExp2C3, f, kExp2C2);
  p = fmaf(p, f, kExp2C1);
  p = fmaf(p, f, kExp2C0);
  // t's integer bits shifted into the exponent field scale p by 2^n.
  return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

}  // namespace jattn
