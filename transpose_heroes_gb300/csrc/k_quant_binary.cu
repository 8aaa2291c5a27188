// Elementwise binary ops on per-tensor quantized operands: dequantize both operands, apply the f32
// op, quantize ("StableHLO Specification": dequantize_op_quantize(op, lhs, rhs, type(result)) for
// add, divide, maximum, minimum, multiply). Same layout everywhere: 16 codes per 16-byte vector;
// otherwise a thread per element with index maps.
#include <algorithm>
#include <cmath>
#include <cooperative_groups.h>

#include "quant_common.cuh"

namespace cg = cooperative_groups;

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

// ---- packed per-tensor kernel (add, maximum, minimum, multiply) -------------------------------------
// Two codes of each operand per f32x2 instruction. A code c becomes the float 1.5*2^23 + (c + 128)
// with one byte permute (the word is first xored with 0x80808080); adding -(1.5*2^23 + 128 + z) gives
// c - z exactly, and the scale product is the dequantized value the spec defines. The op result r is
// quantized with the bracket of the relayout kernel: y = RN(r * RN(1/s)) lies within 2^-23 |y| of
// r / s, and RN(r / s) within 2^-24 more, so when y(1 - 2^-22) and y(1 + 2^-22) round (the magic-constant
// FMA, ties to even) to the same integer, so does RN(r / s). The host admits only parameters that keep
// every |y| below 2^21 (the magic constant's range) and 1/s finite; a word with an undecided code goes
// through the exact per-element path.
struct QbConst {
  float2 sl, sr, zl, zr;  // scales; -(1.5*2^23 + 128 + zero point) of each operand
  float2 io, mo;          // RN(1 / result scale); 1.5*2^23 + result zero point
  int smin, smax;
};

template <int OP>
__device__ __forceinline__ float2 qop2(float2 a, float2 b) {
  if (OP == QOP_ADD) return __fadd2_rn(a, b);
  if (OP == QOP_MULTIPLY) return __fmul2_rn(a, b);
  if (OP == QOP_MAXIMUM) return make_float2(ieee_max(a.x, b.x), ieee_max(a.y, b.y));
  return make_float2(ieee_min(a.x, b.x), ieee_min(a.y, b.y));
}

// Four results for the codes of words a and b; sets `open` when a code is undecided.
template <int OP, bool CLAMP>
__device__ __forceinline__ uint32_t qb_word(uint32_t a, uint32_t b, const QbConst& k, bool& open) {
  const float2 kp = make_float2(1.0f + 0x1p-22f, 1.0f + 0x1p-22f), km = make_float2(1.0f - 0x1p-22f, 1.0f - 0x1p-22f);
  a ^= 0x80808080u;
  b ^= 0x80808080u;
  uint32_t hi = 0u, res = 0u, dw = 0u;
#pragma unroll
  for (int j = 2; j >= 0; j -= 2) {  // codes 2, 3 first: their pack is the upper half of the word
    const float2 ea = make_float2(__uint_as_float(__byte_perm(a, (uint32_t)kMagicBits, 0x7650u | j)),
                                  __uint_as_float(__byte_perm(a, (uint32_t)kMagicBits, 0x7650u | (j + 1))));
    const float2 eb = make_float2(__uint_as_float(__byte_perm(b, (uint32_t)kMagicBits, 0x7650u | j)),
                                  __uint_as_float(__byte_perm(b, (uint32_t)kMagicBits, 0x7650u | (j + 1))));
    const float2 ra = __fmul2_rn(k.sl, __fadd2_rn(ea, k.zl));
    const float2 rb = __fmul2_rn(k.sr, __fadd2_rn(eb, k.zr));
    const float2 y = __fmul2_rn(qop2<OP>(ra, rb), k.io);
    const float2 tp = __ffma2_rn(y, kp, k.mo), tm = __ffma2_rn(y, km, k.mo);
    dw |= (__float_as_uint(tp.x) ^ __float_as_uint(tm.x)) | (__float_as_uint(tp.y) ^ __float_as_uint(tm.y));
    int q0 = __float_as_int(tp.x) - kMagicBits, q1 = __float_as_int(tp.y) - kMagicBits;
    if (CLAMP) {
      q0 = min(max(q0, k.smin), k.smax);
      q1 = min(max(q1, k.smin), k.smax);
    }
    if (j == 2) asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, 0;" : "=r"(hi) : "r"(q1), "r"(q0));
    else asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(res) : "r"(q1), "r"(q0), "r"(hi));
  }
  open = dw != 0u;
  return res;
}

template <int OP, bool CLAMP>
__global__ void __launch_bounds__(256) quant_binary_pk_kernel(QuantBinaryPlan p, QbConst k) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nv = p.n / 16;
  const uint4* l = reinterpret_cast<const uint4*>(p.lhs);
  const uint4* r = reinterpret_cast<const uint4*>(p.rhs);
  uint4* o = reinterpret_cast<uint4*>(p.out);
  constexpr int kU = 2;  // vector pairs in flight per thread
  for (int64_t v0 = tid; v0 < nv; v0 += kU * stride) {
    uint4 a[kU], b[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < nv) {
        a[u] = __ldg(l + v);
        b[u] = __ldg(r + v);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < nv) {
        const uint32_t wa[4] = {a[u].x, a[u].y, a[u].z, a[u].w}, wb[4] = {b[u].x, b[u].y, b[u].z, b[u].w};
        uint32_t res[4];
        bool open[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) res[m] = qb_word<OP, CLAMP>(wa[m], wb[m], k, open[m]);
        if (open[0] | open[1] | open[2] | open[3]) {  // rare: the exact definition decides those words
#pragma unroll
          for (int m = 0; m < 4; ++m)
            if (open[m]) res[m] = qbin4<OP>(wa[m], wb[m], p);
        }
        o[v] = make_uint4(res[0], res[1], res[2], res[3]);
      }
    }
  }
  for (int64_t e = nv * 16 + tid; e < p.n; e += stride) p.out[e] = (int8_t)qbin<OP>(p.lhs[e], p.rhs[e], p);
}

// The packed kernel's constants, or false when the parameters fall outside its range: finite scales,
// a finite nonzero RN(1/s), and |r / s| < 2^21 for every pair of codes.
static bool qb_pk_consts(const QuantBinaryPlan& p, int op, QbConst& k) {
  const double sl = std::fabs((double)p.ql.scale), sr = std::fabs((double)p.qr.scale);
  const double io = std::fabs((double)p.qo.inv_scale);
  if (!(sl < 1e30 && sr < 1e30 && io < 1e30 && io > 0.0)) return false;
  const double da = 256.0 + std::fabs((double)p.ql.zp), db = 256.0 + std::fabs((double)p.qr.zp);  // |c - z|
  double rmax = 0.0;
  if (op == QOP_ADD) rmax = sl * da + sr * db;
  else if (op == QOP_MULTIPLY) rmax = sl * da * sr * db;
  else if (op == QOP_MAXIMUM || op == QOP_MINIMUM) rmax = std::max(sl * da, sr * db);
  else return false;
  if (!(rmax * io * 1.01 < 2097152.0)) return false;
  auto negm = [](int32_t z) { return -(12582912.0f + 128.0f + (float)z); };  // exact for |z| < 2^22
  if (std::abs((int64_t)p.ql.zp) > 1000000 || std::abs((int64_t)p.qr.zp) > 1000000 || std::abs((int64_t)p.qo.zp) > 1000000)
    return false;
  k.sl = make_float2(p.ql.scale, p.ql.scale);
  k.sr = make_float2(p.qr.scale, p.qr.scale);
  k.zl = make_float2(negm(p.ql.zp), negm(p.ql.zp));
  k.zr = make_float2(negm(p.qr.zp), negm(p.qr.zp));
  k.io = make_float2(p.qo.inv_scale, p.qo.inv_scale);
  const float mo = 12582912.0f + (float)p.qo.zp;
  k.mo = make_float2(mo, mo);
  k.smin = p.qo.smin;
  k.smax = p.qo.smax;
  return true;
}

template <int OP>
static cudaError_t qb_pk_launch(const QuantBinaryPlan& p, const QbConst& k, cudaStream_t s) {
  const bool clamp = k.smin > -128 || k.smax < 127;
  const void* kernel = clamp ? (const void*)quant_binary_pk_kernel<OP, true> : (const void*)quant_binary_pk_kernel<OP, false>;
  int64_t blocks = (p.n / 32 + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * kernel_blocks_per_sm(kernel, 256, 0);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (clamp) quant_binary_pk_kernel<OP, true><<<(unsigned)blocks, 256, 0, s>>>(p, k);
  else quant_binary_pk_kernel<OP, false><<<(unsigned)blocks, 256, 0, s>>>(p, k);
  return cudaGetLastError();
}

// Large same-layout inputs: the result depends on the two codes alone, so it is read from a table of
// all 256 x 256 code pairs (64 KiB of shared memory per block). The blocks of a thread-block cluster
// (8 where they fit) build the table together, each computing its share of the pairs with qbin and
// writing them into every block of the cluster through distributed shared memory; after the cluster
// barrier each block streams 16-byte vectors of both operands and looks every pair up locally. No
// global memory beyond the operands and the result.
constexpr int kQbThreads = 1024;
constexpr int kQbEntries = 1 << 16;
constexpr int64_t kQbTableMinElems = int64_t(1) << 22;

// Four results for the four code pairs of two words; the table index is (lhs byte << 8) | rhs byte.
__device__ __forceinline__ uint32_t qb_lookup4(const uint8_t* lut, uint32_t a, uint32_t b) {
  const uint32_t i01 = __byte_perm(b, a, 0x5140), i23 = __byte_perm(b, a, 0x7362);  // [b0 a0 b1 a1], [b2 a2 b3 a3]
  const uint32_t r0 = lut[i01 & 0xFFFFu], r1 = lut[i01 >> 16], r2 = lut[i23 & 0xFFFFu], r3 = lut[i23 >> 16];
  return r0 | (r1 << 8) | (r2 << 16) | (r3 << 24);
}

template <int OP>
__global__ void __launch_bounds__(kQbThreads, 1) quant_binary_table_kernel(QuantBinaryPlan p) {
  extern __shared__ __align__(16) uint8_t qlut[];  // kQbEntries results
  cg::cluster_group cluster = cg::this_cluster();
  const int nb = (int)cluster.num_blocks(), share = kQbEntries / nb;
  for (int c = 8 * (int)threadIdx.x; c < share; c += 8 * kQbThreads) {
    // this block's share, eight consecutive entries at a time, copied to every block of the cluster
    const int first = (int)cluster.block_rank() * share + c;
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = first + i;
      const int r = qbin<OP>((int)(int8_t)(e >> 8), (int)(int8_t)(e & 0xFF), p);
      w[i >> 2] |= ((uint32_t)r & 0xFFu) << (8 * (i & 3));
    }
    for (int d = 0; d < nb; ++d) *reinterpret_cast<uint2*>(cluster.map_shared_rank(qlut, d) + first) = make_uint2(w[0], w[1]);
  }
  cluster.sync();  // every block's table is complete; no shared-memory access crosses blocks after this
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nv = p.n / 16;
  const uint4* l = reinterpret_cast<const uint4*>(p.lhs);
  const uint4* r = reinterpret_cast<const uint4*>(p.rhs);
  uint4* o = reinterpret_cast<uint4*>(p.out);
  constexpr int kU = 2;  // vector pairs in flight per thread
  for (int64_t v0 = tid; v0 < nv; v0 += kU * stride) {
    uint4 a[kU], b[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < nv) {
        a[u] = __ldg(l + v);
        b[u] = __ldg(r + v);
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < nv)
        o[v] = make_uint4(qb_lookup4(qlut, a[u].x, b[u].x), qb_lookup4(qlut, a[u].y, b[u].y),
                          qb_lookup4(qlut, a[u].z, b[u].z), qb_lookup4(qlut, a[u].w, b[u].w));
    }
  }
  for (int64_t e = nv * 16 + tid; e < p.n; e += stride)
    p.out[e] = (int8_t)qlut[((uint32_t)(uint8_t)p.lhs[e] << 8) | (uint8_t)p.rhs[e]];
}

template <int OP>
static cudaError_t qb_table_launch(const QuantBinaryPlan& p, cudaStream_t s) {
  const size_t smem = kQbEntries;
  auto kernel = quant_binary_table_kernel<OP>;
  int cs = 0, clusters = 0;
  table_cluster_shape((const void*)kernel, kQbThreads, smem, &cs, &clusters);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(cs * (clusters > 0 ? clusters : 1)), 1, 1);
  cfg.blockDim = dim3(kQbThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <int OP>
static cudaError_t qb_launch(const QuantBinaryPlan& p, cudaStream_t s) {
  const bool same = p.lmap.identity && p.rmap.identity && p.omap.identity;
  const bool aligned = ((uintptr_t)p.lhs % 16 == 0) && ((uintptr_t)p.rhs % 16 == 0) && ((uintptr_t)p.out % 16 == 0);
  QbConst k;
  if (OP != QOP_DIVIDE && same && aligned && qb_pk_consts(p, OP, k))
    return qb_pk_launch<OP == QOP_DIVIDE ? QOP_ADD : OP>(p, k, s);  // (no packed divide)
  if (same && aligned && p.n >= kQbTableMinElems) return qb_table_launch<OP>(p, s);
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
