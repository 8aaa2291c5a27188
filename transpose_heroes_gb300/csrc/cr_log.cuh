// Correctly rounded single-precision natural logarithm for sm_103a.
//
// The spec defines log as the IEEE-754 log of the element type ("StableHLO Specification", section
// "log"); IEEE-754 recommends correct rounding, which makes the f32 result unique, so the fused
// transpose can be bit-exact. The implementation is written from the mathematics:
//
//   x = 2^e * m, m in [OFF, 2*OFF) with OFF ~ 0.706; c = the centre of m's table interval,
//   log x = e*ln2 + log(c) + log1p(r),  r = m * inv_c - 1 (exact: see gen_log_table.py),
//   log1p(r) = r - r^2/2 + r^3 * (1/3 - r/4 + r^2/5 - r^3/6) + O(r^7).
//
// Stage 1 evaluates this sum in float-float arithmetic (Fast2Sum, exact FMA products), then applies a
// rounding test (Ziv's strategy) with the error bound 2^-44 |y| + 2^-23 |r|^3: if the error interval
// around the float-float value contains no rounding boundary of f32, the leading float is the
// correctly rounded result. The bound is at least twice the largest error of the evaluation over every
// positive normal f32 input (an exhaustive check; the input set is finite). Otherwise (probability
// ~2^-19 per element) stage 2 recomputes log x with double-double sums to better than 2^-70 relative
// and rounds that.
// Special operands (0, negative, subnormal, inf, NaN, exactly 1) also take stage 2.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "log_table.inc"

namespace hlo {

// ------------------------------------------------------------------------------------------------
// double-double helpers (Dekker / Knuth error-free transformations)
// ------------------------------------------------------------------------------------------------
struct dd {
  double hi, lo;
};

__device__ __forceinline__ dd dd_two_sum(double a, double b) {
  double s = __dadd_rn(a, b);
  double bb = __dsub_rn(s, a);
  double err = __dadd_rn(__dsub_rn(a, __dsub_rn(s, bb)), __dsub_rn(b, bb));
  return {s, err};
}

__device__ __forceinline__ dd dd_fast_two_sum(double a, double b) {  // requires |a| >= |b|
  double s = __dadd_rn(a, b);
  return {s, __dsub_rn(b, __dsub_rn(s, a))};
}

__device__ __forceinline__ dd dd_two_prod(double a, double b) {
  double p = __dmul_rn(a, b);
  return {p, __fma_rn(a, b, -p)};
}

__device__ __forceinline__ dd dd_add(dd x, dd y) {  // accurate: two_sum on both components
  dd s = dd_two_sum(x.hi, y.hi);
  dd t = dd_two_sum(x.lo, y.lo);
  s.lo = __dadd_rn(s.lo, t.hi);
  s = dd_fast_two_sum(s.hi, s.lo);
  s.lo = __dadd_rn(s.lo, t.lo);
  return dd_fast_two_sum(s.hi, s.lo);
}

// Rounds the double-double value y (|y.lo| <= ulp(y.hi)/2) to the nearest f32, ties to even.
__device__ __forceinline__ float dd_to_f32_rn(dd y) {
  float f = __double2float_rn(y.hi);
  double d = __dadd_rn(__dsub_rn(y.hi, (double)f), y.lo);  // y - f; the first difference is exact
  if (d == 0.0) return f;
  float nb = d > 0 ? __int_as_float(__float_as_int(f) + ((f >= 0.0f) ? 1 : -1))
                   : __int_as_float(__float_as_int(f) + ((f > 0.0f) ? -1 : 1));
  if (f == 0.0f) nb = d > 0 ? 1e-45f : -1e-45f;
  double half = __dmul_rn(__dsub_rn((double)nb, (double)f), 0.5);  // signed half gap towards d
  double ad = fabs(d), ah = fabs(half);
  if (ad < ah) return f;
  if (ad > ah) return nb;
  return (__float_as_uint(f) & 1u) ? nb : f;  // exact tie: even significand
}

// ------------------------------------------------------------------------------------------------
// Stage 2 (inputs stage 1 cannot round, and every special operand). Same reduction as stage 1,
// x = 2^e m, r = m * inv_c - 1 exact, and
//   log x = e*ln2 + log(c) + r - r^2/2 + r^3 P(r),   P(r) = 1/3 - r/4 + r^2/5 - ... - r^7/10,
// |r| < 2^-8.5, so the truncation (r^11/11) stays below 2^-94. FP64 is a slow pipe on this part (one
// warp instruction per 64 cycles), so the common case takes ~30 double operations:
//   A = e*LN2_HI + LOGC_HI is exact (ln 2 on the 2^-44 grid, log(c) on the 2^-45 grid, |e*ln2| < 2^7);
//   S + E = A + r exactly (Fast2Sum: A = 0 or |A| > |r|);
//   M = -r^2/2 + r^3 P(r) + e*LN2_LO + LOGC_LO in double (error < 2^-70.9 absolute, and relative to r^2
//   when A = 0); yh + yl = S + (E + M) exactly.
// The total error is below 2^-61.5 |y|; when no f32 rounding boundary lies within 2^-60 |y| of
// yh + yl, the nearer float is the answer. Otherwise (about 2^-16 of these calls) the double-double
// evaluation below, accurate to better than 2^-100, decides.
// ------------------------------------------------------------------------------------------------
static __device__ __noinline__ float cr_logf_dd(int e, double r, int i) {
  const double r2 = __dmul_rn(r, r);                             // exact
  double p = -0.1;
  p = __fma_rn(p, r, 1.0 / 9.0);
  p = __fma_rn(p, r, -0.125);
  p = __fma_rn(p, r, 1.0 / 7.0);
  p = __fma_rn(p, r, -1.0 / 6.0);
  p = __fma_rn(p, r, 0.2);
  p = __fma_rn(p, r, -0.25);
  p = __fma_rn(p, r, 1.0 / 3.0);
  const double t = __dmul_rn(__dmul_rn(r2, r), p);               // r^3 P(r)
  dd l1 = dd_two_sum(r, __dmul_rn(-0.5, r2));                    // r - r^2/2, exact
  l1 = dd_add(l1, {t, 0.0});                                     // log1p(r)
  const double2 lct = kLogC3[i];
  const dd lc = dd_fast_two_sum(lct.x, lct.y);                   // log(c), normalised
  const double ed = (double)e;
  dd el = dd_two_prod(HLO_LN2_DD_HI, ed);                        // e*ln2
  el.lo = __fma_rn(HLO_LN2_DD_LO, ed, el.lo);
  el = dd_fast_two_sum(el.hi, el.lo);
  const dd y = dd_add(dd_add(el, lc), l1);
  return dd_to_f32_rn(y);
}

static __device__ __noinline__ float cr_logf_accurate(float x) {
  uint32_t ix = __float_as_uint(x);
  if (x != x) return x;                                   // NaN stays NaN
  if ((ix & 0x7FFFFFFFu) == 0) return __int_as_float(0xFF800000);  // log(+-0) = -inf
  if (ix >> 31) return __int_as_float(0x7FC00000);        // negative: invalid, quiet NaN
  if (ix == 0x7F800000u) return x;                        // log(+inf) = +inf
  if (ix == 0x3F800000u) return 0.0f;                     // log(1) = +0
  int eadj = 0;
  if (ix < 0x00800000u) {                                 // subnormal: scale into the normal range
    ix = __float_as_uint(x * 8388608.0f);
    eadj = -23;
  }
  const uint32_t tmp = ix - HLO_LOG_OFF;
  const int e = ((int)tmp >> 23) + eadj;
  const int i = (int)((tmp >> HLO_LOG_SHIFT) & (HLO_LOG_NC - 1));
  const float m = __uint_as_float(ix - (tmp & 0xFF800000u));
  const double r = (double)__fmaf_rn(m, kLogCTab[i].x, -1.0f);  // exact by table construction
  const double r2 = __dmul_rn(r, r);                             // exact
  double p = -0.1;
  p = __fma_rn(p, r, 1.0 / 9.0);
  p = __fma_rn(p, r, -0.125);
  p = __fma_rn(p, r, 1.0 / 7.0);
  p = __fma_rn(p, r, -1.0 / 6.0);
  p = __fma_rn(p, r, 0.2);
  p = __fma_rn(p, r, -0.25);
  p = __fma_rn(p, r, 1.0 / 3.0);
  const double t = __dmul_rn(__dmul_rn(r2, r), p);               // r^3 P(r)
  const double2 lc = kLogC3[i];
  const double ed = (double)e;
  const double A = __fma_rn(ed, HLO_LN2_DD_HI, lc.x);            // exact
  const double S = __dadd_rn(A, r);
  const double E = __dsub_rn(r, __dsub_rn(S, A));
  const double M = __fma_rn(-0.5, r2, __dadd_rn(t, __fma_rn(ed, HLO_LN2_DD_LO, lc.y)));
  const double L = __dadd_rn(E, M);
  const double yh = __dadd_rn(S, L);
  const double yl = __dsub_rn(L, __dsub_rn(yh, S));
  // f = nearest float to yh; d = (yh + yl) - f; h = half the gap from f to its neighbour towards d
  const float f = __double2float_rn(yh);
  const double d = __dadd_rn(__dsub_rn(yh, (double)f), yl);
  if (d == 0.0) return f;
  const uint32_t fb = __float_as_uint(f);
  const float nb = __uint_as_float((d > 0.0) == (f > 0.0f) ? fb + 1u : fb - 1u);
  const double h = __dmul_rn(__dsub_rn((double)nb, (double)f), 0.5);
  const double margin = __dmul_rn(fabs(yh), 0x1p-60);
  const double ad = fabs(d), ah = fabs(h);
  if (ad < __dsub_rn(ah, margin)) return f;
  if (ad > __dadd_rn(ah, margin)) return nb;
  return cr_logf_dd(e, r, i);
}

// ------------------------------------------------------------------------------------------------
// Stage 1. ctab/etab may point to shared or global copies of kLogCTab / kLogETab. Returns the
// correctly rounded log when ok is set; ok is cleared for special operands and for results whose
// rounding the error bound cannot decide (stage 2 must then be used).
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ float cr_logf_fast(float x, const float4* __restrict__ ctab,
                                              const float2* __restrict__ etab, bool& ok) {
  const uint32_t ix = __float_as_uint(x);
  const bool normal = ix - 0x00800000u < 0x7F000000u;  // positive normal
  const uint32_t tmp = ix - HLO_LOG_OFF;
  const int e = normal ? (int)tmp >> 23 : 0;
  const uint32_t i = (tmp >> HLO_LOG_SHIFT) & (HLO_LOG_NC - 1);
  const float m = __uint_as_float(ix - (tmp & 0xFF800000u));
  const float4 c = ctab[i];                       // inv_c, log c hi, log c lo
  const float2 E = etab[e - HLO_LOG_EMIN];        // e*ln2 hi, lo
  const float r = __fmaf_rn(m, c.x, -1.0f);       // exact by table construction
  // s1 = E_hi + logc_hi: E_hi is 0 or dominates, so Fast2Sum is exact
  const float s1 = __fadd_rn(E.x, c.y);
  const float e1 = __fsub_rn(c.y, __fsub_rn(s1, E.x));
  // s2 = s1 + r: s1 is 0 or |s1| >= |r| (table check / |e*ln2| - |log c| > |r|)
  const float s2 = __fadd_rn(s1, r);
  const float e2 = __fsub_rn(r, __fsub_rn(s2, s1));
  // -r^2/2 split exactly into qh + ql
  const float hr = -0.5f * r;
  const float qh = __fmul_rn(hr, r);
  const float ql = __fmaf_rn(hr, r, -qh);
  const float s3 = __fadd_rn(s2, qh);
  const float e3 = __fsub_rn(qh, __fsub_rn(s3, s2));
  // r^3 (1/3 - r/4 + r^2/5 - r^3/6)
  float p = __fmaf_rn(r, -0.16666667f, 0.2f);
  p = __fmaf_rn(r, p, -0.25f);
  p = __fmaf_rn(r, p, 0.33333334f);
  const float r3 = __fmul_rn(__fmul_rn(r, r), r);
  float lo = __fmaf_rn(r3, p, ql);
  lo = __fadd_rn(lo, __fadd_rn(E.y, c.z));
  lo = __fadd_rn(lo, __fadd_rn(__fadd_rn(e1, e2), e3));
  const float yh = __fadd_rn(s3, lo);
  const float yl = __fsub_rn(lo, __fsub_rn(yh, s3));
  // rounding test: boundary at half an ulp of yh; powers of two and y = 0 are left to stage 2
  const float err = __fmaf_rn(fabsf(yh), 0x1p-44f, __fmul_rn(fabsf(r3), 0x1p-23f));
  const uint32_t yb = __float_as_uint(yh);
  const float half_ulp = __uint_as_float((yb & 0x7F800000u) - (24u << 23));
  ok = normal & (__fadd_rn(fabsf(yl), err) < half_ulp) & ((yb & 0x007FFFFFu) != 0u);
  return yh;
}

__device__ __forceinline__ float cr_logf(float x, const float4* __restrict__ ctab, const float2* __restrict__ etab) {
  bool ok;
  const float y = cr_logf_fast(x, ctab, etab, ok);
  return ok ? y : cr_logf_accurate(x);
}

// ------------------------------------------------------------------------------------------------
// Packed f32x2 arithmetic through CUDA's float2 intrinsics (one instruction per pair of lanes, each
// lane rounded to nearest even, never contracted).
// ------------------------------------------------------------------------------------------------
namespace f2 {
__device__ __forceinline__ float2 pk(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ void upk(float2 r, float& a, float& b) {
  a = r.x;
  b = r.y;
}
__device__ __forceinline__ float2 splat(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 add(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 sub(float2 a, float2 b) { return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a); }  // a - b, one rounding
__device__ __forceinline__ float2 mul(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
}  // namespace f2

// ------------------------------------------------------------------------------------------------
// First pass, two elements at a time: 32-interval table (three 32-float arrays, so a warp's lookups
// hit distinct banks), e*ln2 from exact products:
//   log x = S + err + rest,  S + err = A + r exactly (Fast2Sum),  A = e*LN2_A + log(c)_hi (exact),
//   rest = r^2 (-1/2 + r/3 - r^2/4 + r^3/5) + (e*LN2_B + log(c)_lo)   in f32   (|r| < 2^-5.6).
// With lo = RN(err + rest), the errors (truncation r^6/6 < 2^-36.2 of the alternating series, the
// roundings of r^2, of the polynomial and of rest ~2^-36.3 each, the table and LN2_B terms below 2^-36
// for all exponents, lo's rounding ~2^-36.2) stay under b = 2^-33.5 less the rounding of lo +- b
// (< 2^-37): a step-for-step emulation of these operations over every positive normal float gives
// |log x - (S + lo)| <= 2^-34.13 (2^-34.40 with the r^6 term kept, which costs one more packed FMA
// per pair). Rounding test by monotonicity of round-to-nearest: if S + (lo - b)
// and S + (lo + b) round to the same float, every value between them, the exact log among them,
// rounds to it. About 2% of inputs in [0.5, 2) (most of those near 1) and every special operand
// are left open (ok = false) for cr_logf.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void cr_logf_first2(float x0, float x1, const float* __restrict__ tinv,
                                               const float* __restrict__ thi, const float* __restrict__ tlo,
                                               float& y0, float& y1, bool& ok0, bool& ok1) {
  const uint32_t ix0 = __float_as_uint(x0), ix1 = __float_as_uint(x1);
  const bool n0 = ix0 - 0x00800000u < 0x7F000000u, n1 = ix1 - 0x00800000u < 0x7F000000u;
  const uint32_t t0 = ix0 - HLO_LOG1_OFF, t1 = ix1 - HLO_LOG1_OFF;
  const uint32_t i0 = (t0 >> HLO_LOG1_SHIFT) & 31u, i1 = (t1 >> HLO_LOG1_SHIFT) & 31u;
  const float m0 = __uint_as_float(ix0 - (t0 & 0xFF800000u)), m1 = __uint_as_float(ix1 - (t1 & 0xFF800000u));
  // e as a float through the 1.5*2^23 constant (|e| < 2^22): bits 0x4B400000 + e, minus 1.5*2^23
  const float eb0 = __int_as_float(0x4B400000 + ((int)t0 >> 23));
  const float eb1 = __int_as_float(0x4B400000 + ((int)t1 >> 23));
  const float2 EF = f2::add(f2::pk(eb0, eb1), f2::splat(-12582912.0f));
  const float2 R = f2::fma(f2::pk(m0, m1), f2::pk(tinv[i0], tinv[i1]), f2::splat(-1.0f));  // exact
  const float2 A = f2::fma(EF, f2::splat(HLO_LOG1_LN2_A), f2::pk(thi[i0], thi[i1]));        // exact
  const float2 S = f2::add(A, R);                       // Fast2Sum: A = 0 or |A| >= |r|
  const float2 ERR = f2::sub(R, f2::sub(S, A));
  float2 P = f2::fma(R, f2::splat(0.2f), f2::splat(-0.25f));
  P = f2::fma(R, P, f2::splat(0.33333334f));
  P = f2::fma(R, P, f2::splat(-0.5f));
  const float2 B = f2::fma(EF, f2::splat(HLO_LOG1_LN2_B), f2::pk(tlo[i0], tlo[i1]));
  const float2 REST = f2::fma(f2::mul(R, R), P, B);
  const float2 LO = f2::add(ERR, REST);
  const float bound = 0x1.6a09e6p-34f;                  // 2^-33.5
  const float2 YP = f2::add(S, f2::add(LO, f2::splat(bound)));
  const float2 YM = f2::add(S, f2::sub(LO, f2::splat(bound)));
  y0 = YP.x;
  y1 = YP.y;
  ok0 = n0 & (YP.x == YM.x);
  ok1 = n1 & (YP.y == YM.y);
}

// The same first pass for four values, with the tables' addresses known at compile time (static shared
// memory: `tab` holds the 32 inv_c, then the 32 log(c)_hi, then the 32 log(c)_lo) and the test for
// positive normal operands made once for all four: the table offset is read straight from the bits,
// (t >> (HLO_LOG1_SHIFT - 2)) & (31 << 2), and a block with any special operand leaves all four open.
// Returns the four candidates in y and the settled ones as bits 0..3 of the result.
__device__ __forceinline__ uint32_t cr_logf_first4(const float4 x, const float (&tab)[96], float4& y) {
  const uint32_t ix[4] = {__float_as_uint(x.x), __float_as_uint(x.y), __float_as_uint(x.z), __float_as_uint(x.w)};
  const int mn = min(min((int)ix[0], (int)ix[1]), min((int)ix[2], (int)ix[3]));
  const int mx = max(max((int)ix[0], (int)ix[1]), max((int)ix[2], (int)ix[3]));
  const bool normal = (mn >= 0x00800000) & (mx < 0x7F800000);
  float ym[4], yp[4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t t0 = ix[2 * h] - HLO_LOG1_OFF, t1 = ix[2 * h + 1] - HLO_LOG1_OFF;
    const uint32_t b0 = (t0 >> (HLO_LOG1_SHIFT - 2)) & (31u << 2), b1 = (t1 >> (HLO_LOG1_SHIFT - 2)) & (31u << 2);
    const char* tb = reinterpret_cast<const char*>(tab);
    const float m0 = __uint_as_float(ix[2 * h] - (t0 & 0xFF800000u)), m1 = __uint_as_float(ix[2 * h + 1] - (t1 & 0xFF800000u));
    const float eb0 = __int_as_float(0x4B400000 + ((int)t0 >> 23));
    const float eb1 = __int_as_float(0x4B400000 + ((int)t1 >> 23));
    const float2 EF = f2::add(f2::pk(eb0, eb1), f2::splat(-12582912.0f));
    const float2 INV = f2::pk(*reinterpret_cast<const float*>(tb + b0), *reinterpret_cast<const float*>(tb + b1));
    const float2 HI = f2::pk(*reinterpret_cast<const float*>(tb + 128 + b0), *reinterpret_cast<const float*>(tb + 128 + b1));
    const float2 LOT = f2::pk(*reinterpret_cast<const float*>(tb + 256 + b0), *reinterpret_cast<const float*>(tb + 256 + b1));
    const float2 R = f2::fma(f2::pk(m0, m1), INV, f2::splat(-1.0f));  // exact
    const float2 A = f2::fma(EF, f2::splat(HLO_LOG1_LN2_A), HI);       // exact
    const float2 S = f2::add(A, R);                                     // Fast2Sum: A = 0 or |A| >= |r|
    const float2 ERR = f2::sub(R, f2::sub(S, A));
    float2 P = f2::fma(R, f2::splat(0.2f), f2::splat(-0.25f));
    P = f2::fma(R, P, f2::splat(0.33333334f));
    P = f2::fma(R, P, f2::splat(-0.5f));
    const float2 B = f2::fma(EF, f2::splat(HLO_LOG1_LN2_B), LOT);
    const float2 REST = f2::fma(f2::mul(R, R), P, B);
    const float2 LO = f2::add(ERR, REST);
    const float bound = 0x1.6a09e6p-34f;  // 2^-33.5, as in cr_logf_first2
    const float2 YP = f2::add(S, f2::add(LO, f2::splat(bound)));
    const float2 YM = f2::add(S, f2::sub(LO, f2::splat(bound)));
    yp[2 * h] = YP.x;
    yp[2 * h + 1] = YP.y;
    ym[2 * h] = YM.x;
    ym[2 * h + 1] = YM.y;
  }
  y = make_float4(yp[0], yp[1], yp[2], yp[3]);
  if (!normal) return 0u;
  return (yp[0] == ym[0] ? 1u : 0u) | (yp[1] == ym[1] ? 2u : 0u) | (yp[2] == ym[2] ? 4u : 0u) |
         (yp[3] == ym[3] ? 8u : 0u);
}

// Loads the 32-entry first-pass table into shared memory (three arrays of 32 floats).
__device__ __forceinline__ void load_log1_tables(float* s_inv, float* s_hi, float* s_lo) {
  for (int i = threadIdx.x; i < 32; i += blockDim.x) {
    s_inv[i] = kLog1Inv[i];
    s_hi[i] = kLog1Hi[i];
    s_lo[i] = kLog1Lo[i];
  }
}

// Loads the tables into shared memory (called by all threads of a block, followed by a barrier).
__device__ __forceinline__ void load_log_tables(float4* sc, float2* se) {
  for (int i = threadIdx.x; i < HLO_LOG_NC; i += blockDim.x) sc[i] = kLogCTab[i];
  for (int i = threadIdx.x; i < HLO_LOG_NE; i += blockDim.x) se[i] = kLogETab[i];
}

}  // namespace hlo
