// Uniform quantization helpers shared by the quantized kernels ("StableHLO Quantization": real =
// scale * (q - zero_point); quantize = clamp(round_nearest_even(real / scale) + zero_point)).
#pragma once
#include "device_common.cuh"

namespace hlo {

constexpr float kMagic = 12582912.0f;      // 1.5 * 2^23: x + kMagic rounds x to an integer (|x| < 2^22)
constexpr int kMagicBits = 0x4B400000;     // bit pattern of kMagic

// real = scale * (q - zero_point): exact integer difference, exact int -> float (|d| <= 255 < 2^22
// through the magic constant), one f32 multiply.
__device__ __forceinline__ float dequant(int code, float scale, int zp) {
  const int d = code - zp;
  const float df = __fsub_rn(__int_as_float(kMagicBits + d), kMagic);
  return __fmul_rn(scale, df);
}

// The exact definition: clamp(rint(real / scale) + zp), IEEE f32 division, NaN -> zero point.
static __device__ __noinline__ int quant_code_exact(float real, float scale, int zp, int smin, int smax) {
  if (real != real) return zp;
  const float y = __fdiv_rn(real, scale);
  float q = __fadd_rn(rintf(y), (float)zp);
  q = fminf(fmaxf(q, (float)smin), (float)smax);
  return (int)q;
}

// Same result, fast: with inv = RN(1/scale) the product real*inv is within 2^-23 relative of
// real/scale, and the IEEE quotient within 2^-24; when the product is farther than 2^-22 (relative)
// from the nearest half-integer, all three round to the same integer, which the magic-constant add
// produces (ties to even). Otherwise, or out of range / NaN, the exact definition decides.
__device__ __forceinline__ int quant_code(float real, float scale, float inv, int zp, int smin, int smax) {
  const float y = __fmul_rn(real, inv);
  const float t = __fadd_rn(y, kMagic);
  const float f = __fsub_rn(y, __fsub_rn(t, kMagic));
  const float ay = fabsf(y);
  if (!(ay < 4194304.0f) || fabsf(__fsub_rn(fabsf(f), 0.5f)) <= __fmul_rn(ay, 0x1p-22f))
    return quant_code_exact(real, scale, zp, smin, smax);
  const int q = (__float_as_int(t) - kMagicBits) + zp;
  return min(max(q, smin), smax);
}

}  // namespace hlo
