// Elementwise binary ops on per-tensor quantized operands: dequantize both operands, apply the f32
// op, quantize ("StableHLO Specification": dequantize_op_quantize(op, lhs, rhs, type(result)) for
// add, divide, maximum, minimum, multiply). Same layout everywhere: 16 codes per 16-byte vector;
// otherwise a thread per element with index maps.
#include "quant_common.cuh"

namespace hlo {

enum QOp : int { QOP_ADD = 0, QOP_DIVIDE = 1, QOP_MAXIMUM = 2, QOP_MINIMUM = 3, QOP_MULTIPLY = 4 };

// IEEE-754 minimum: NaN propagates; -0 < +0.
__device__ __forceinline__ float ieee_min(float a, float b) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

template <int OP>
__device__ __forceinline__ float qop(float a, float b) {
  if (OP == QOP_ADD) return __fadd_rn(a, b);
  if (OP == QOP_DIVIDE) return __fdiv_rn(a, b);
  if (OP == QOP_MAXIMUM) return ieee_max(a, b);
  if (OP == QOP_MINIMUM) return ieee_min(a, b);
  return __fmul_rn(a, b);
}

template <int OP>
__device__ __forceinline__ int qbin(int a, int b, const QuantBinaryPlan& p) {
  const float r = qop<OP>(dequant(a, p.ql.scale, p.ql.zp), dequant(b, p.qr.scale, p.qr.zp));
  return quant_code(r, p.qo.scale, p.qo.inv_scale, p.qo.zp, p.qo.smin, p.qo.smax);
}

template <int OP>
__device__ __forceinline__ uint32_t qbin4(uint32_t a, uint32_t b, const QuantBinaryPlan& p) {
  uint32_t o = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = qbin<OP>((int)(int8_t)(a >> (8 * j)), (int)(int8_t)(b >> (8 * j)), p);
    o |= ((uint32_t)r & 0xFFu) << (8 * j);
  }
  return o;
}

template <int OP>
__global__ void __launch_bounds__(256) quant_binary_vec_kernel(QuantBinaryPlan p) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nv = p.n / 16;
  const uint4* l = reinterpret_cast<const uint4*>(p.lhs);
  const uint4* r = reinterpret_cast<const uint4*>(p.rhs);
  uint4* o = reinterpret_cast<uint4*>(p.out);
  for (int64_t i = tid; i < nv; i += stride) {
    const uint4 a = __ldg(l + i), b = __ldg(r + i);
    o[i] = make_uint4(qbin4<OP>(a.x, b.x, p), qbin4<OP>(a.y, b.y, p), qbin4<OP>(a.z, b.z, p), qbin4<OP>(a.w, b.w, p));
  }
  for (int64_t e = nv * 16 + tid; e < p.n; e += stride) p.out[e] = (int8_t)qbin<OP>(p.lhs[e], p.rhs[e], p);
}

template <int OP>
__global__ void __launch_bounds__(256) quant_binary_map_kernel(QuantBinaryPlan p) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < p.n; i += stride)
    p.out[map_index(p.omap, i)] = (int8_t)qbin<OP>(p.lhs[map_index(p.lmap, i)], p.rhs[map_index(p.rmap, i)], p);
}

template <int OP>
static cudaError_t qb_launch(const QuantBinaryPlan& p, cudaStream_t s) {
  const bool same = p.lmap.identity && p.rmap.identity && p.omap.identity;
  const bool aligned = ((uintptr_t)p.lhs % 16 == 0) && ((uintptr_t)p.rhs % 16 == 0) && ((uintptr_t)p.out % 16 == 0);
  const int64_t per = same && aligned ? 16 : 1;
  int64_t blocks = (p.n / per + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (same && aligned) quant_binary_vec_kernel<OP><<<(unsigned)blocks, 256, 0, s>>>(p);
  else quant_binary_map_kernel<OP><<<(unsigned)blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_quant_binary(const QuantBinaryPlan& p, cudaStream_t s) {
  if (p.n == 0) return cudaSuccess;
  switch (p.op) {
    case QOP_ADD: return qb_launch<QOP_ADD>(p, s);
    case QOP_DIVIDE: return qb_launch<QOP_DIVIDE>(p, s);
    case QOP_MAXIMUM: return qb_launch<QOP_MAXIMUM>(p, s);
    case QOP_MINIMUM: return qb_launch<QOP_MINIMUM>(p, s);
    default: return qb_launch<QOP_MULTIPLY>(p, s);
  }
}

}  // namespace hlo
