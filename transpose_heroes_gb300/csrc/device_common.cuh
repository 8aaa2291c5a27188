// Device helpers shared by the kernel translation units: element conversion, rounding to 16-bit
// float types, the elementwise ops of a chain, and the reduce bodies.
#pragma once
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "cr_exp.cuh"
#include "cr_log.cuh"
#include "hlo_internal.h"

namespace hlo {

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) { return __half2float(__ushort_as_half(h)); }
__device__ __forceinline__ uint16_t f32_to_f16_bits(float f) { return __half_as_ushort(__float2half_rn(f)); }

__device__ __forceinline__ float load_as_f32(const void* p, int dt, int64_t i) {
  switch (dt) {
    case F32: return __ldg(reinterpret_cast<const float*>(p) + i);
    case BF16: return bf16_bits_to_f32(__ldg(reinterpret_cast<const unsigned short*>(p) + i));
    case F16: return f16_bits_to_f32(__ldg(reinterpret_cast<const unsigned short*>(p) + i));
    case S8: return (float)__ldg(reinterpret_cast<const signed char*>(p) + i);
    case S32: return (float)__ldg(reinterpret_cast<const int*>(p) + i);
  }
  return 0.f;
}

// Stores v (already representable in dt for the float types) converting with round-to-nearest-even.
__device__ __forceinline__ void store_from_f32(void* p, int dt, int64_t i, float v) {
  switch (dt) {
    case F32: reinterpret_cast<float*>(p)[i] = v; break;
    case BF16: reinterpret_cast<uint16_t*>(p)[i] = f32_to_bf16_bits(v); break;
    case F16: reinterpret_cast<uint16_t*>(p)[i] = f32_to_f16_bits(v); break;
    case S8: reinterpret_cast<int8_t*>(p)[i] = (int8_t)__float2int_rn(v); break;
    case S32: reinterpret_cast<int32_t*>(p)[i] = __float2int_rn(v); break;
  }
}

__device__ __forceinline__ float round_to_dt(float v, int dt) {
  if (dt == BF16) return bf16_bits_to_f32(f32_to_bf16_bits(v));
  if (dt == F16) return f16_bits_to_f32(f32_to_f16_bits(v));
  return v;
}

// exp(x) = 2^(x log2 e) on the SFU. Used only as the last op before an add-combine of a float
// reduction: RN(x log2 e) carries a relative error of at most 2^-24 |x log2 e| <= 2^-17 for the finite
// range |x| < 89, so a term's relative error stays below about 2^-17 (plus the SFU's own ~2^-22) --
// inside the add reduction's tolerance of 1e-5 sum|terms|. Results below 2^-126 are flushed to zero
// (an absolute error under 2^-126 per term). Never used where a value is rounded afterwards for a
// bit-exact result (max bodies, transposes, elementwise chains).
__device__ __forceinline__ float fast_exp(float x) {
  float t = __fmul_rn(x, 1.4426950408889634f);
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(t));
  return y;
}

// IEEE-754 maximum: NaN propagates; -0 < +0.
__device__ __forceinline__ float ieee_max(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// The reduce body and its identity.
template <int KIND>
__device__ __forceinline__ float combine(float a, float b) {
  if (KIND == RED_ADD) return __fadd_rn(a, b);
  return ieee_max(a, b);
}
template <int KIND>
__device__ __forceinline__ float identity() {
  return KIND == RED_ADD ? 0.0f : __int_as_float(0xFF800000);
}
__device__ __forceinline__ float combine_rt(int kind, float a, float b) {
  return kind == RED_ADD ? __fadd_rn(a, b) : ieee_max(a, b);
}

// Shared log tables: either staged in shared memory by the kernel or read from global memory.
struct LogTab {
  const float4* c;
  const float2* e;
};
__device__ __forceinline__ LogTab global_log_tables() { return {kLogCTab, kLogETab}; }

// Correct rounding into a 16-bit float type from an f32 approximation y of f(x) with an error of at
// most 2 f32 ulps: if y - 2 ulp and y + 2 ulp round alike, so does f(x) (rounding is monotone).
// Returns false (and leaves r unset) when they do not, or when y sits next to 0, the subnormals or
// the top of the range, where the ulp test is not valid.
__device__ __forceinline__ bool round16_settled(float y, int dt, float& r) {
  const uint32_t b = __float_as_uint(y), a = b & 0x7FFFFFFFu;
  if (a >= 0x7F800000u) {  // inf, NaN
    r = y;
    return true;
  }
  if (a < 0x00800002u || a > 0x7F7FFFFDu) return false;
  const float v = round_to_dt(y, dt);
  if (round_to_dt(__uint_as_float(b - 2u), dt) != v || round_to_dt(__uint_as_float(b + 2u), dt) != v) return false;
  r = v;
  return true;
}

// A double rounded once into a 16-bit float type: round to odd into f32 (truncate, then set the last
// bit if anything was cut off), then to nearest even; f32 keeps at least 2 bits more than the 16-bit
// significand, so the second rounding cannot go wrong.
__device__ __forceinline__ float round16_from_double(double d, int dt) {
  float t = __double2float_rz(d);
  if ((double)t != d && !isinf(t)) t = __uint_as_float(__float_as_uint(t) | 1u);
  return round_to_dt(t, dt);
}

// exp / tanh / log correctly rounded into bf16 or f16 for a 16-bit input: the f32 result (CUDA's expf
// and tanhf are within 2 ulp, cr_logf within half an ulp) settles almost every element; the rest
// (about 2^-14 of them) take CUDA's double exp/tanh/log (within 1 double ulp), rounded once.
static __device__ __noinline__ float exp_round16_slow(float x, int dt) { return round16_from_double(exp((double)x), dt); }
static __device__ __noinline__ float tanh_round16_slow(float x, int dt) { return round16_from_double(tanh((double)x), dt); }
static __device__ __noinline__ float log_round16_slow(float x, int dt) { return round16_from_double(log((double)x), dt); }

// exp as a chain op: correctly rounded to f32, or (r16) to the 16-bit element type dt, where CUDA's
// expf settles almost every element.
__device__ __forceinline__ float chain_exp(float v, bool r16, int dt) {
  float r;
  if (!r16) return cr_expf(v);
  return round16_settled(expf(v), dt, r) ? r : exp_round16_slow(v, dt);
}

__device__ __forceinline__ float chain_log(float v, bool r16, int dt, const float4* c, const float2* e) {
  float r;
  if (!r16) return cr_logf(v, c, e);
  return round16_settled(cr_logf(v, c, e), dt, r) ? r : log_round16_slow(v, dt);
}

__device__ __forceinline__ float chain_tanh(float v, bool r16, int dt) {
  float r;
  if (!r16) return cr_tanhf(v);
  return round16_settled(tanhf(v), dt, r) ? r : tanh_round16_slow(v, dt);
}

// The same three, out of line: the kernels that interpret chains at run time call one shared copy
// instead of inlining all three evaluations at every use (which multiplies code size and build time).
static __device__ __noinline__ float chain_exp_call(float v, bool r16, int dt) { return chain_exp(v, r16, dt); }
static __device__ __noinline__ float chain_log_call(float v, bool r16, int dt, const float4* c, const float2* e) {
  return chain_log(v, r16, dt, c, e);
}
static __device__ __noinline__ float chain_tanh_call(float v, bool r16, int dt) { return chain_tanh(v, r16, dt); }

// One elementwise op of a chain, every result correctly rounded (exp, log, tanh) or exact.
__device__ __forceinline__ float apply_op(int op, float v, float b, float x, float imm, bool r16, int dt,
                                          const LogTab& lt) {
  switch (op) {
    case OP_EXP: return chain_exp_call(v, r16, dt);
    case OP_LOG: return chain_log_call(v, r16, dt, lt.c, lt.e);
    case OP_TANH: return chain_tanh_call(v, r16, dt);
    case OP_ABS: return fabsf(v);
    case OP_NEG: return -v;
    case OP_ADD_BCAST: return __fadd_rn(v, b);
    case OP_ADD_CONST: return __fadd_rn(v, imm);
    case OP_MUL_CONST: return __fmul_rn(v, imm);
    case OP_ADD_IN: return __fadd_rn(v, x);
    case OP_MUL_IN: return __fmul_rn(v, x);
  }
  return v;
}

// Runtime-interpreted chain (used by the general kernels). boff = offset of the broadcast element.
// With round16 every op result is rounded to the 16-bit element type: f32 arithmetic on two 16-bit
// values followed by one rounding equals the correctly rounded 16-bit operation (f32 has at least
// 2p + 2 significand bits for p = 8 and 11).
__device__ __forceinline__ float apply_chain_rt(const Chain& c, float v, int64_t boff, const LogTab& lt) {
  const float x = v;
  const bool r16 = c.round16 && (c.dt == BF16 || c.dt == F16);
  for (int k = 0; k < c.n; ++k) {
    const int op = c.op[k];
    float b = 0.f;
    if (op == OP_ADD_BCAST) b = load_as_f32(c.bptr, c.bdt, boff);
    v = apply_op(op, v, b, x, c.imm[k], r16, c.dt, lt);
    if (c.round16) v = round_to_dt(v, c.dt);
  }
  return v;
}

__host__ __device__ inline bool chain_has_bcast_dev(const Chain& c) {
  for (int k = 0; k < c.n; ++k)
    if (c.op[k] == OP_ADD_BCAST) return true;
  return false;
}

__device__ __forceinline__ bool chain_has_log(const Chain& c) {
  for (int k = 0; k < c.n; ++k)
    if (c.op[k] == OP_LOG) return true;
  return false;
}

}  // namespace hlo
