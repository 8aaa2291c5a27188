// Device helpers shared by the kernel translation units: element conversion, rounding to 16-bit
// float types, the elementwise ops of a chain, and the reduce bodies.
#pragma once
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

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

// exp(x) = 2^(x log2 e) on the SFU: relative error ~2^-21, used where the hero is a float reduction
// whose tolerance absorbs it.
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

// One elementwise op. FAST_EXP selects the SFU exp (reductions) or CUDA's expf (elsewhere).
template <bool FAST_EXP>
__device__ __forceinline__ float apply_op(int op, float v, float b, const LogTab& lt) {
  switch (op) {
    case OP_EXP: return FAST_EXP ? fast_exp(v) : expf(v);
    case OP_LOG: return cr_logf(v, lt.c, lt.e);
    case OP_ABS: return fabsf(v);
    case OP_NEG: return -v;
    case OP_ADD_BCAST: return __fadd_rn(v, b);
  }
  return v;
}

// Runtime-interpreted chain (used by the general kernels). boff = offset of the broadcast element.
template <bool FAST_EXP>
__device__ __forceinline__ float apply_chain_rt(const Chain& c, float v, int64_t boff, const LogTab& lt) {
  for (int k = 0; k < c.n; ++k) {
    int op = c.op[k];
    float b = 0.f;
    if (op == OP_ADD_BCAST) b = load_as_f32(c.bptr, c.bdt, boff);
    v = apply_op<FAST_EXP>(op, v, b, lt);
    if (c.round16) v = round_to_dt(v, c.dt);
  }
  return v;
}

__device__ __forceinline__ bool chain_has_log(const Chain& c) {
  for (int k = 0; k < c.n; ++k)
    if (c.op[k] == OP_LOG) return true;
  return false;
}

}  // namespace hlo
