// Correctly rounded f32 exp and tanh ("StableHLO Specification", sections "exponential" and "tanh":
// the IEEE-754 function of the element type; rounding to nearest even of the exact value).
//
// Stage 1: CUDA's double exp, documented within 1 double ulp, rounded once to f32. That rounding is
// the correct one unless the double lies within 3 double ulps of an f32 rounding boundary (a
// midpoint between two floats), which happens for about 2^-26 of the arguments.
// Stage 2 (those, and NaN): a double-double evaluation after Tang ("Table-driven implementation of
// the exponential function in IEEE floating-point arithmetic", ACM TOMS 15(2), 1989):
//   k = rint(64 x / ln2) = 64 e + j,  r = x - k ln2/64 (as a double-double, exactly up to 2^-94),
//   exp x = 2^e * 2^(j/64) * exp(r),  exp(r) = 1 + r + r^2/2 + r^3 P(r),
// P the Taylor polynomial to r^6/7! (|r| < 2^-7.4, so the truncation is below 2^-97), with every
// rounding error below 2^-74 relative; the nearer float of that value is returned.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "cr_log.cuh"  // double-double helpers
#include "exp_table.inc"

namespace hlo {

// exp(a) as a double-double (about 2^-74 relative), for a double a that is an f32 value in
// [-104, 89] (or twice one in [-52, 44.5]).
__device__ __forceinline__ dd exp_dd(double a) {
  const double kd = rint(__dmul_rn(a, HLO_EXP_INV64_LN2));
  const int k = (int)kd;
  const double b = __fma_rn(-kd, HLO_EXP_L1, a);  // exact: k L1 has at most 53 bits, |b| < 2^-6
  const dd p2 = dd_two_prod(kd, HLO_EXP_L2);       // k L2 exactly
  dd r = dd_two_sum(b, -p2.hi);
  r.lo = __dsub_rn(__dsub_rn(r.lo, p2.lo), __dmul_rn(kd, HLO_EXP_L3));
  r = dd_fast_two_sum(r.hi, r.lo);
  const double rh = r.hi, rl = r.lo;
  // r^3 (1/3! + r/4! + r^2/5! + r^3/6! + r^4/7!) in double (rl's share is below 2^-75)
  double p = 1.0 / 5040.0;
  p = __fma_rn(p, rh, 1.0 / 720.0);
  p = __fma_rn(p, rh, 1.0 / 120.0);
  p = __fma_rn(p, rh, 1.0 / 24.0);
  p = __fma_rn(p, rh, 1.0 / 6.0);
  const double q = __dmul_rn(__dmul_rn(__dmul_rn(rh, rh), rh), p);
  // 1 + rh + rh^2/2 exactly as double-doubles, then the small terms
  const dd sq = dd_two_prod(rh, rh);
  const dd s1 = dd_fast_two_sum(1.0, rh);
  const dd s2 = dd_two_sum(s1.hi, __dmul_rn(sq.hi, 0.5));
  double small = __dadd_rn(s1.lo, s2.lo);
  small = __dadd_rn(small, rl);
  small = __dadd_rn(small, __fma_rn(rh, rl, __dmul_rn(sq.lo, 0.5)));
  small = __dadd_rn(small, q);
  const dd e = dd_fast_two_sum(s2.hi, small);
  // times 2^(j/64) (double-double) and 2^(k >> 6)
  const double2 t = kExpT[k & 63];
  const dd pr = dd_two_prod(t.x, e.hi);
  const double lo = __dadd_rn(pr.lo, __fma_rn(t.x, e.lo, __dmul_rn(t.y, e.hi)));
  dd y = dd_fast_two_sum(pr.hi, lo);
  const double scale = __hiloint2double((1023 + (k >> 6)) << 20, 0);  // 2^e, e in [-163, 128]
  y.hi = __dmul_rn(y.hi, scale);
  y.lo = __dmul_rn(y.lo, scale);
  return y;
}

static __device__ __noinline__ float cr_expf_dd(float x) {
  if (x != x) return x;                               // NaN
  if (x > 89.0f) return __int_as_float(0x7F800000);  // exp > 2^128: +inf
  if (x < -104.0f) return 0.0f;                       // exp < 2^-150: rounds to +0
  const dd y = exp_dd((double)x);
  const float f = __double2float_rn(y.hi);
  if (isinf(f)) return f;
  return dd_to_f32_rn(y);
}

// Distance test shared by exp and tanh: true if the double y (within 1 double ulp of the exact value)
// rounds to the same f32 as the exact value, i.e. y is more than 3 double ulps from a boundary.
__device__ __forceinline__ bool f32_rounding_settled(double y) {
  const double a = fabs(y);
  if (a >= 0x1p-126) {  // normal f32 range (and inf): the boundary is at 2^28 in the 29 low bits
    const uint32_t low = (uint32_t)__double_as_longlong(y) & 0x1FFFFFFFu;
    return low - (0x10000000u - 3u) > 6u;
  }
  if (a >= 0.0) {  // subnormal or zero f32: boundaries at odd multiples of 2^-150
    const double s = __dmul_rn(a, 0x1p149);  // exact
    const double fr = __dsub_rn(s, floor(s));
    return fabs(__dsub_rn(fr, 0.5)) > __dmul_rn(s, 0x1p-50);
  }
  return false;  // NaN
}

__device__ __forceinline__ float cr_expf(float x) {
  const double y = exp((double)x);
  return f32_rounding_settled(y) ? __double2float_rn(y) : cr_expf_dd(x);
}

// ------------------------------------------------------------------------------------------------
// Correctly rounded f32 tanh ("StableHLO Specification", section "tanh"), the same way: CUDA's double
// tanh (within 1 double ulp) rounded once unless it sits within 3 double ulps of an f32 boundary; then
// a double-double value decides. tanh is odd, so |x| is evaluated and the sign restored:
//   |x| < 2^-6:      x + x^3 P(x^2), the Taylor series to x^13 (truncation below 2^-78 relative);
//   2^-6 <= |x| < 10: (t - 1) / (t + 1) with t = exp(2|x|) as a double-double (t - 1 >= 2^-5, so the
//                    subtraction costs at most 5 of its 74 bits), the quotient to double-double;
//   |x| >= 10:       1 - tanh|x| < 2^-28, which rounds to 1.
// ------------------------------------------------------------------------------------------------
static __device__ __noinline__ float cr_tanhf_dd(float x) {
  if (x != x) return x;
  const float ax = fabsf(x);
  if (ax >= 10.0f) return copysignf(1.0f, x);
  dd y;
  const double a = (double)ax;
  if (ax < 0x1p-6f) {
    const double z = __dmul_rn(a, a);
    double p = 21844.0 / 6081075.0;  // x^13
    p = __fma_rn(p, z, -1382.0 / 155925.0);
    p = __fma_rn(p, z, 62.0 / 2835.0);
    p = __fma_rn(p, z, -17.0 / 315.0);
    p = __fma_rn(p, z, 2.0 / 15.0);
    p = __fma_rn(p, z, -1.0 / 3.0);
    const dd a3 = dd_two_prod(z, a);  // z = a^2 rounded: its error is below 2^-53 a^3, ~2^-66 a
    const dd z2 = dd_two_prod(a, a);
    const double cube_lo = __fma_rn(z2.lo, a, a3.lo);  // a^3 = (z2.hi + z2.lo) a
    const dd c = dd_two_prod(a3.hi, p);
    y = dd_fast_two_sum(a, c.hi);
    y.lo = __dadd_rn(y.lo, __fma_rn(cube_lo, p, c.lo));
    y = dd_fast_two_sum(y.hi, y.lo);
  } else {
    const dd t = exp_dd(__dmul_rn(2.0, a));
    const dd num = dd_add(t, {-1.0, 0.0});
    const dd den = dd_add(t, {1.0, 0.0});
    // num / den: q0 = num.hi / den.hi, then one correction with the exact remainder
    const double q0 = __ddiv_rn(num.hi, den.hi);
    const dd m = dd_two_prod(q0, den.hi);
    const double rem = __dsub_rn(__dadd_rn(__dsub_rn(__dsub_rn(num.hi, m.hi), m.lo), num.lo), __dmul_rn(q0, den.lo));
    const double q1 = __ddiv_rn(rem, den.hi);
    y = dd_fast_two_sum(q0, q1);
  }
  const float f = dd_to_f32_rn(y);
  return x < 0.0f ? -f : f;
}

__device__ __forceinline__ float cr_tanhf(float x) {
  if (fabsf(x) < 0x1p-126f) return x;  // zero and subnormals: |tanh x - x| is far below half an ulp
  const double y = tanh((double)x);
  return f32_rounding_settled(y) ? __double2float_rn(y) : cr_tanhf_dd(x);
}

}  // namespace hlo
