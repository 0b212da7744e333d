// bf16_round.cuh — the correctly rounded RMSNorm output shared by the norm
// kernels and the QKV-projection epilogue: x_hat = bf16(g x r) with
// r = (mean x^2 + eps)^(-1/2), rounded to the bf16 value nearest the exact
// real product (device code only).
#pragma once
#include <cstdint>

namespace jattn {

constexpr float kEps = 1e-6f;

// --- correctly rounded x_hat ------------------------------------------------
// x_hat is the bf16 value nearest to the exact real g x r.  The fp32 value
// y = (g x) r computed with the fp32 sum of squares and rsqrtf is within 10.5
// fp32 units in the last place of the exact product (first order in
// u = 2^-24): the squares of bf16 values are exact and the sum takes at most
// 8 roundings of nonnegative terms (3 per packed accumulator, 1 to join them,
// log2(d/8) <= 4 across lanes): 8u; the mean and eps add u; rsqrtf is good
// to 2 ulp (4u) and halves the relative error of its argument (4.5u); the
// two products add u each.  Rounding y to bf16 is therefore exact unless y
// lies within 16 fp32 ulps of a bf16 midpoint (low 16 bits 0x8000): the
// window test takes the 32 values 0x8000 - 16 .. 0x8000 + 15.  Those elements
// are rounded from a double-float r accurate to about 2^-44: the row's sum
// of squares by error-free additions, one Newton step from rsqrtf, and an
// error-free product, with the remainder's sign breaking the midpoint.  A
// warp takes that path when any of its lanes has such an element (about one
// element in two thousand).
constexpr uint32_t kTieWindow = 32;
constexpr float kEpsLo = static_cast<float>(1e-6 - static_cast<double>(1e-6f));

// Knuth's TwoSum and Dekker's Fast2Sum (|a| >= |b|), with the _rn intrinsics
// so that nothing is contracted or reassociated.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  e = __fsub_rn(b, __fsub_rn(s, a));
}


// (rh, rl) = (m + eps)^(-1/2) as a double-float, from the double-float sum
// (s, c) of the row's squares and inv_d = 1/d (a power of two: exact
// scaling).
__device__ __forceinline__ void rsqrt_mean_eps_df(float s, float c, float inv_d, float& rh, float& rl) {
  float mh, ml, e1;
  two_sum(__fmul_rn(s, inv_d), kEps, mh, e1);
  fast_two_sum(mh, __fadd_rn(__fadd_rn(__fmul_rn(c, inv_d), kEpsLo), e1), mh, ml);
  // r = r0 (1 - t)^(-1/2) with 1 - t = m r0^2, t of order 2^-22.
  const float r0 = rsqrtf(mh);
  const float ph = __fmul_rn(r0, r0), pl = __fmaf_rn(r0, r0, -ph);
  const float qh = __fmul_rn(mh, ph);
  const float ql = __fmaf_rn(ml, ph, __fmaf_rn(mh, pl, __fmaf_rn(mh, ph, -qh)));
  const float t = __fsub_rn(__fsub_rn(1.f, qh), ql);
  fast_two_sum(r0, __fmul_rn(r0, __fmul_rn(t, __fmaf_rn(0.375f, t, 0.5f))), rh, rl);
}

// A float whose round-to-nearest-even bf16 conversion is the bf16 value
// nearest to g x (rh + rl).
__device__ __forceinline__ float round_bf16_df(float g, float x, float rh, float rl) {
  const float yh = __fmul_rn(g, x), yl = __fmaf_rn(g, x, -yh);
  float zh = __fmul_rn(yh, rh);
  float zl = __fmaf_rn(yl, rh, __fmaf_rn(yh, rl, __fmaf_rn(yh, rh, -zh)));
  fast_two_sum(zh, zl, zh, zl);
  const uint32_t b = __float_as_uint(zh);
  if ((b & 0xFFFFu) == 0x8000u && zl != 0.f) {
    const bool up = (zl > 0.f) == (zh > 0.f);  // away from zero
    return __uint_as_float((b & 0xFFFF0000u) + (up ? 0x10000u : 0u));
  }
  return zh;  // not a midpoint, or an exact one (ties to even)
}

__device__ __forceinline__ bool near_bf16_midpoint(float y) {
  return ((__float_as_uint(y) + (kTieWindow / 2 - 0x8000u)) & (0xFFFFu & ~(kTieWindow - 1))) == 0u;
}

}  // namespace jattn
