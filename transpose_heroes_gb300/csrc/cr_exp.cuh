// Correctly rounded f32 exp and tanh ("StableHLO Specification", sections "exponential" and "tanh":
// the IEEE-754 function of the element type; rounding to nearest even of the exact value).
//
// Stage 1 (cr_expf): a float-float evaluation in f32 with a rounding test, below.
// Stage 2: CUDA's double exp, documented within 1 double ulp, rounded once to f32. That rounding is
// the correct one unless the double lies within 3 double ulps of an f32 rounding boundary (a
// midpoint between two floats), which happens for about 2^-26 of the arguments.
// Stage 3 (those, and NaN): a double-double evaluation after Tang ("Table-driven implementation of
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

static __device__ __noinline__ float cr_expf_double(float x) {
  const double y = exp((double)x);
  return f32_rounding_settled(y) ? __double2float_rn(y) : cr_expf_dd(x);
}

// First pass in f32 for arguments with a normal, finite result (about 1 in 2^11 of them stays open):
//   k = rint(64 x / ln2) through the 1.5*2^23 constant, r1 = x - k L1f exactly (k L1f is exact and the
//   difference fits 24 bits for every f32 in range, checked exhaustively), r = rh + rl = r1 - k L2f -
//   k L3f (the k L2f product split exactly by FMA, the sum by TwoSum),
//   exp(r) - 1 = rh + pe,  pe = rh^2 (1/2 + rh/6 + rh^2/24) + rl (1 + rh)   (truncation < 2^-44),
//   y = yh + yl = 2^(j/64) (1 + rh + pe), with 2^(j/64) = Th + Tl and Th rh split exactly by FMA,
//   exp x = 2^(k >> 6) y.
// Every rounding error sums to under 2^-36.5 absolute (y < 2.02; 2^-37.2 in an emulation over 4.2 M
// arguments); with b = 2^-35 the rounding is decided by monotonicity: if yh + (yl - b) and
// yh + (yl + b) round to the same float, so does y. Scaling by 2^e is exact in the normal range.
// The reduction of both f32 passes: k = rint(64 x / ln2), x - k ln2/64 = rh + rl to about 2^-54.
__device__ __forceinline__ void expf_reduce(float x, int& k, float& rh, float& rl) {
  const float t = __fmaf_rn(x, HLO_EXPF_INV64_LN2, 12582912.0f);
  k = __float_as_int(t) - 0x4B400000;
  const float kf = __fsub_rn(t, 12582912.0f);
  const float r1 = __fmaf_rn(-kf, HLO_EXPF_L1, x);  // exact
  const float p2h = __fmul_rn(kf, HLO_EXPF_L2);
  const float p2l = __fmaf_rn(kf, HLO_EXPF_L2, -p2h);  // k L2f = p2h + p2l exactly
  rh = __fsub_rn(r1, p2h);                               // TwoSum(r1, -p2h)
  const float bb = __fsub_rn(rh, r1);
  rl = __fadd_rn(__fsub_rn(r1, __fsub_rn(rh, bb)), __fsub_rn(-p2h, bb));
  rl = __fmaf_rn(-kf, HLO_EXPF_L3, __fsub_rn(rl, p2l));
}

__device__ __forceinline__ void expf_ff(float x, float& yh, float& yl, int& e) {
  int k;
  float rh, rl;
  expf_reduce(x, k, rh, rl);
  float q = __fmaf_rn(rh, 0x1.555556p-5f, 0x1.555556p-3f);  // 1/24, 1/6
  q = __fmaf_rn(rh, q, 0.5f);
  float pe = __fmaf_rn(__fmul_rn(rh, rh), q, rl);
  pe = __fmaf_rn(rl, rh, pe);
  const float2 T = __ldg(&kExpTf[k & 63]);
  const float ah = __fmul_rn(T.x, rh);
  const float al = __fmaf_rn(T.x, rh, -ah);
  float lo = __fmaf_rn(T.x, pe, T.y);
  lo = __fadd_rn(__fmaf_rn(T.y, rh, lo), al);
  yh = __fadd_rn(T.x, ah);  // Fast2Sum: Th >= 1 > |ah|
  yl = __fadd_rn(__fsub_rn(ah, __fsub_rn(yh, T.x)), lo);
  e = k >> 6;
}

// Second f32 pass, for the arguments the first leaves open (about 1 in 2000), before any FP64 work
// (FP64 issues at 1/64 of the FP32 rate on this part). The same reduction, then
//   E = exp(r) - 1 = r + r^2/2 + r^3/6 + r^4/24 + r^5/120   (|r| < 2^-7.5: the r^6 term is below 2^-54)
// as an unnormalised pair: r^2/2 from the exact FMA split of rh^2 plus rh rl, the r^3 rh-rl cross term
// (rh^2 rl / 2), and rh^3 (1/6 + rh/24 + rh^2/120) in f32 (below 2^-25.2, relative error under 2^-22);
// then y = (Th + Tl)(1 + E) with the Th E_hi product split exactly by FMA and Th + (Th E_hi)_hi summed
// exactly (Th >= 1 > |Th E_hi|). Error terms: E's roundings under 2^-46.4, the table pair under 2^-48
// relative, y's low-part roundings under 2^-45.5: all under 2^-44.4 for y < 2.02. With b = 2^-43 the
// monotone rounding test of the first pass decides all but about 2^-19 of these arguments; those take
// the double path.
static __device__ __noinline__ float cr_expf_stage2(float x) {
  int k;
  float rh, rl;
  expf_reduce(x, k, rh, rl);
  const float ph = __fmul_rn(rh, rh);
  const float pl = __fmaf_rn(rh, rh, -ph);  // rh^2 = ph + pl exactly
  const float h = __fmul_rn(0.5f, ph), hl = __fmul_rn(0.5f, pl);  // exact
  float q = __fmaf_rn(rh, 0x1.111112p-7f, 0x1.555556p-5f);       // 1/120, 1/24
  q = __fmaf_rn(rh, q, 0x1.555556p-3f);                            // 1/6
  const float c = __fmul_rn(__fmul_rn(ph, rh), q);                 // r^3/6 + r^4/24 + r^5/120
  const float sh = __fadd_rn(rh, h);                               // Fast2Sum: |rh| > |h|
  const float sl = __fsub_rn(h, __fsub_rn(sh, rh));
  float t = __fmaf_rn(rh, rl, rl);                                 // rl (1 + rh)
  t = __fmaf_rn(h, rl, t);                                         // + rh^2 rl / 2
  t = __fadd_rn(t, hl);
  t = __fadd_rn(t, c);
  const float el = __fadd_rn(sl, t);                               // E = sh + el
  const float2 T = __ldg(&kExpTf[k & 63]);
  const float qh = __fmul_rn(T.x, sh);
  const float qe = __fmaf_rn(T.x, sh, -qh);                        // Th sh = qh + qe exactly
  const float yh = __fadd_rn(T.x, qh);                             // Fast2Sum: Th >= 1 > |qh|
  const float ye = __fsub_rn(qh, __fsub_rn(yh, T.x));
  float lo = __fmaf_rn(T.y, sh, T.y);                              // Tl (1 + E_hi)
  lo = __fmaf_rn(T.x, el, lo);                                     // + Th E_lo
  lo = __fadd_rn(lo, qe);
  const float yl = __fadd_rn(ye, lo);
  const float yp = __fadd_rn(yh, __fadd_rn(yl, 0x1p-43f));
  const float ym = __fadd_rn(yh, __fsub_rn(yl, 0x1p-43f));
  if (yp == ym) return __fmul_rn(yp, __int_as_float((127 + (k >> 6)) << 23));
  return cr_expf_double(x);
}

__device__ __forceinline__ float cr_expf(float x) {
  if (x > -87.0f && x < 88.5f) {
    float yh, yl;
    int e;
    expf_ff(x, yh, yl, e);
    const float yp = __fadd_rn(yh, __fadd_rn(yl, 0x1p-35f));
    const float ym = __fadd_rn(yh, __fsub_rn(yl, 0x1p-35f));
    if (yp == ym) return __fmul_rn(yp, __int_as_float((127 + e) << 23));
    return cr_expf_stage2(x);
  }
  return cr_expf_double(x);
}

// The passes after the first, for an argument the first pass left open (or outside its range).
static __device__ __noinline__ float cr_expf_rest(float x) {
  return (x > -87.0f && x < 88.5f) ? cr_expf_stage2(x) : cr_expf_double(x);
}

// The first pass for two arguments at once in packed f32x2 arithmetic (the same operations as
// expf_ff and the rounding test of cr_expf, each lane rounded alike). ok0 / ok1 report a settled
// result; an open argument, or one outside (-87, 88.5), is the caller's to finish with cr_expf_rest.
__device__ __forceinline__ void cr_expf_first2(float x0, float x1, float& y0, float& y1, bool& ok0, bool& ok1) {
  const float2 X = f2::pk(x0, x1);
  const float2 T = f2::fma(X, f2::splat(HLO_EXPF_INV64_LN2), f2::splat(12582912.0f));
  const int k0 = __float_as_int(T.x) - 0x4B400000, k1 = __float_as_int(T.y) - 0x4B400000;
  const float2 KF = f2::add(T, f2::splat(-12582912.0f));
  const float2 R1 = f2::fma(KF, f2::splat(-HLO_EXPF_L1), X);                  // exact
  const float2 P2H = f2::mul(KF, f2::splat(HLO_EXPF_L2));
  const float2 NP2H = f2::mul(P2H, f2::splat(-1.0f));                         // exact
  const float2 P2L = f2::fma(KF, f2::splat(HLO_EXPF_L2), NP2H);               // k L2f = p2h + p2l
  const float2 RH = f2::add(R1, NP2H);                                        // TwoSum(r1, -p2h)
  const float2 BB = f2::sub(RH, R1);
  float2 RL = f2::add(f2::sub(R1, f2::sub(RH, BB)), f2::sub(NP2H, BB));
  RL = f2::fma(KF, f2::splat(-HLO_EXPF_L3), f2::sub(RL, P2L));
  float2 Q = f2::fma(RH, f2::splat(0x1.555556p-5f), f2::splat(0x1.555556p-3f));  // 1/24, 1/6
  Q = f2::fma(RH, Q, f2::splat(0.5f));
  float2 PE = f2::fma(f2::mul(RH, RH), Q, RL);
  PE = f2::fma(RL, RH, PE);
  const float2 t0 = __ldg(&kExpTf[k0 & 63]), t1 = __ldg(&kExpTf[k1 & 63]);
  const float2 TX = f2::pk(t0.x, t1.x), TY = f2::pk(t0.y, t1.y);
  const float2 AH = f2::mul(TX, RH);
  const float2 AL = f2::fma(TX, RH, f2::mul(AH, f2::splat(-1.0f)));
  float2 LO = f2::fma(TX, PE, TY);
  LO = f2::add(f2::fma(TY, RH, LO), AL);
  const float2 YH = f2::add(TX, AH);  // Fast2Sum: Th >= 1 > |ah|
  const float2 YL = f2::add(f2::sub(AH, f2::sub(YH, TX)), LO);
  const float2 YP = f2::add(YH, f2::add(YL, f2::splat(0x1p-35f)));
  const float2 YM = f2::add(YH, f2::sub(YL, f2::splat(0x1p-35f)));
  const float2 Y = f2::mul(YP, f2::pk(__int_as_float((127 + (k0 >> 6)) << 23), __int_as_float((127 + (k1 >> 6)) << 23)));
  y0 = Y.x;
  y1 = Y.y;
  ok0 = (x0 > -87.0f) & (x0 < 88.5f) & (YP.x == YM.x);
  ok1 = (x1 > -87.0f) & (x1 < 88.5f) & (YP.y == YM.y);
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

static __device__ __noinline__ float cr_tanhf_double(float x) {
  const double y = tanh((double)x);
  return f32_rounding_settled(y) ? __double2float_rn(y) : cr_tanhf_dd(x);
}

// First pass in f32 (a = |x|, sign restored at the end), then the rounding test of cr_expf:
//   a < 2^-4:  tanh a = a - a^3/3 + a^5 P(a^2), P = 2/15 - 17 a^2/315 + 62 a^4/2835 - 1382 a^6/155925
//              (truncation below 2^-45 a); a^3/3 as an f32 pair (a^2, a^3 split by FMA, 1/3 as an
//              f32 pair), the a^5 P term in f32: error below 2^-40 a; test bound a 2^-37.
//   2^-4 <= a < 9.05: tanh a = 1 - 2/(t + 1), t = exp(2a) as an f32 pair from expf_ff (error below
//              2^-36.5 t); 2/(t + 1) = q0 + q1 with q0 the IEEE quotient of the high parts and q1 from
//              its exact remainder; 1 - q0 split exactly. Error below 2^-37.3 absolute; bound 2^-35.5.
//   a >= 9.05: 1 - tanh a < 2^-25.1, so tanh rounds to 1.
__device__ __forceinline__ float cr_tanhf(float x) {
  const float a = fabsf(x);
  if (a < 0x1p-126f) return x;  // zero and subnormals: |tanh x - x| is far below half an ulp
  if (a >= 9.05f) return a == a ? copysignf(1.0f, x) : x;
  float th, tl, b;
  if (a < 0x1p-4f) {
    const float a2h = __fmul_rn(a, a), a2l = __fmaf_rn(a, a, -a2h);
    const float a3h = __fmul_rn(a, a2h);
    const float a3l = __fmaf_rn(a, a2l, __fmaf_rn(a, a2h, -a3h));
    const float ch = __fmul_rn(a3h, 0x1.555556p-2f);
    const float cl = __fmaf_rn(a3l, 0x1.555556p-2f, __fmaf_rn(a3h, -0x1.555556p-27f, __fmaf_rn(a3h, 0x1.555556p-2f, -ch)));
    float p = __fmaf_rn(a2h, -0x1.226e36p-7f, 0x1.664f48p-6f);
    p = __fmaf_rn(a2h, p, -0x1.ba1ba2p-5f);
    p = __fmaf_rn(a2h, p, 0x1.111112p-3f);
    const float t5 = __fmul_rn(__fmul_rn(a3h, a2h), p);
    th = __fsub_rn(a, ch);  // Fast2Sum: a > a^3/3
    tl = __fadd_rn(__fsub_rn(__fsub_rn(a, th), ch), __fsub_rn(t5, cl));
    b = __fmul_rn(a, 0x1p-37f);
  } else {
    float yh, yl;
    int e;
    expf_ff(__fmul_rn(2.0f, a), yh, yl, e);
    const float sc = __int_as_float((127 + e) << 23);  // 2^e, e in [0, 26]
    const float eh = __fmul_rn(yh, sc), el = __fmul_rn(yl, sc);
    const float d1 = __fadd_rn(eh, 1.0f);  // Fast2Sum: eh >= 1
    const float d2 = __fadd_rn(__fsub_rn(1.0f, __fsub_rn(d1, eh)), el);
    const float dh = __fadd_rn(d1, d2);  // renormalised (el is not below half an ulp of eh)
    const float dl = __fsub_rn(d2, __fsub_rn(dh, d1));
    const float q0 = __fdiv_rn(2.0f, dh);
    const float r = __fmaf_rn(-q0, dl, __fmaf_rn(-q0, dh, 2.0f));  // 2 - q0 dh is exact
    const float q1 = __fmul_rn(r, __fmul_rn(q0, 0.5f));
    th = __fsub_rn(1.0f, q0);  // Fast2Sum: 1 > q0
    tl = __fsub_rn(__fsub_rn(__fsub_rn(1.0f, th), q0), q1);
    b = 0x1.6a09e6p-36f;  // 2^-35.5
  }
  const float yp = __fadd_rn(th, __fadd_rn(tl, b));
  const float ym = __fadd_rn(th, __fsub_rn(tl, b));
  if (yp == ym) return x < 0.0f ? -yp : yp;
  return cr_tanhf_double(x);
}

}  // namespace hlo
