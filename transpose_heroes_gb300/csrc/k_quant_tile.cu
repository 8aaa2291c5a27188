// Quantized relayout hero kernel ("StableHLO Quantization": real = scale * (q - zero_point), per-tensor
// or per-axis; "XLA Shapes and Layout", section "Layout"):
//
//  quant_tile_kernel    -- s8 [n0, n1] row-major -> column-major with dequantize / quantize fused:
//                          128 x 128-byte tiles, 16-byte loads, an XOR-swizzled shared tile read back
//                          4 bytes at a time, 4x4 byte transposes in registers, 16-byte stores.
//  quant_tma_kernel     -- the same tiles for whole-tile shapes with per-tensor output parameters: each
//                          tile (and its per-axis input parameters) arrives by tensor / bulk copies
//                          into a ring of shared-memory stages, so the loads of later tiles overlap
//                          the arithmetic and the stores of earlier ones.
#include "async_copy.cuh"
#include "device_common.cuh"
#include "quant_common.cuh"

namespace hlo {

// ---------------------------------------------------------------------------------------------
// quantization
// ---------------------------------------------------------------------------------------------
constexpr int kQT = 128;  // tile edge in bytes

struct __align__(16) QuantSmem {
  float sin_[kQT];   // input scale per tile row (axis 0) or column (axis 1)
  int zin[kQT];
  float sout[kQT];   // output scale per tile row or column
  float inv[kQT];    // RN(1 / output scale)
  int zout[kQT];
  int zinm[kQT];     // kMagicBits - input zero point: code + zinm = bits of (1.5*2^23 + code - zp)
  float nzin[kQT];   // -(1.5*2^23 + 128 + input zero point), exact
  float mout[kQT];   // 1.5*2^23 + output zero point, exact
};

// Ragged or unaligned tile, byte by byte (kept out of line: it is rare and large).
__device__ __noinline__ void quant_tile_ragged(const QuantTilePlan& p, int64_t i0, int64_t j0, uint8_t* bt,
                                               const QuantSmem& q) {
  const int t = threadIdx.x;
  for (int e = t; e < kQT * kQT; e += blockDim.x) {
    const int row = e / kQT, col = e % kQT;
    const int64_t i = i0 + row, j = j0 + col;
    if (i < p.n0 && j < p.n1) {
      const int code = (int)p.in[i * p.n1 + j];
      float sin = p.qin.scale;
      int zin = p.qin.zp;
      if (p.qin.axis == 0) { sin = q.sin_[row]; zin = q.zin[row]; }
      if (p.qin.axis == 1) { sin = q.sin_[col]; zin = q.zin[col]; }
      float real = dequant(code, sin, zin);
      if (p.ops.n) real = apply_chain_rt(p.ops, real, 0, global_log_tables());
      float sout = p.qout.scale, inv = p.qout.inv_scale;
      int zout = p.qout.zp;
      if (p.qout.axis == 0) { sout = q.sout[row]; inv = q.inv[row]; zout = q.zout[row]; }
      if (p.qout.axis == 1) { sout = q.sout[col]; inv = q.inv[col]; zout = q.zout[col]; }
      bt[col * kQT + row] = (uint8_t)quant_code(real, sout, inv, zout, p.qout.smin, p.qout.smax);
    }
  }
  __syncthreads();
  for (int e = t; e < kQT * kQT; e += blockDim.x) {
    const int col = e / kQT, row = e % kQT;
    const int64_t i = i0 + row, j = j0 + col;
    if (i < p.n0 && j < p.n1) p.out[j * p.n0 + i] = (int8_t)bt[col * kQT + row];
  }
}

template <int QIN, int QOUT, bool OPS>
__device__ __forceinline__ void quant_params(int row, int jl, const QuantTilePlan& p, const QuantSmem& q, float& sin,
                                             int& zin, float& sout, float& inv, int& zout) {
  sin = QIN == 0 ? q.sin_[row] : QIN == 1 ? q.sin_[jl] : p.qin.scale;
  zin = QIN == 0 ? q.zin[row] : QIN == 1 ? q.zin[jl] : p.qin.zp;
  sout = QOUT == 0 ? q.sout[row] : QOUT == 1 ? q.sout[jl] : p.qout.scale;
  inv = QOUT == 0 ? q.inv[row] : QOUT == 1 ? q.inv[jl] : p.qout.inv_scale;
  zout = QOUT == 0 ? q.zout[row] : QOUT == 1 ? q.zout[jl] : p.qout.zp;
}

// Dequantize -> [float chain] -> quantize for two codes with float2 arithmetic. The fast path of
// quant_code: y = real * RN(1/scale) is within 2^-22 |y| of the IEEE quotient, so both round to the
// same integer when 0.5 - |y - rint(y)| > 2^-22 |y|. With f = y - rint(y), 0.5 - |f| >= 1/4 - f^2 and
// 2^-22 |y| <= 2^-31 y^2 + 2^-15 (|y| <= (y^2/a + a)/2 with a = 2^8), so it suffices that
// f^2 + 2^-31 y^2 < 1/4 - 2^-15 - 2^-24 (the last term absorbs the roundings of the test). NaN,
// infinities and |y| >= 2^14.5 fail the test as well. Lanes that fail are settled exactly later.
template <bool OPS>
__device__ __forceinline__ void quant_two(int c0, int c1, float2 sin, int zm0, int zm1, float2 inv, int zo0, int zo1,
                                          int smin, int smax, const QuantTilePlan& p, int& q0, int& q1, bool& ok0,
                                          bool& ok1) {
  const float2 magic = make_float2(kMagic, kMagic);
  const float2 df = __fadd2_rn(make_float2(__int_as_float(c0 + zm0), __int_as_float(c1 + zm1)),
                               make_float2(-kMagic, -kMagic));  // exact code - zero point
  float2 real = __fmul2_rn(sin, df);
  if (OPS) {
    real.x = apply_chain_rt(p.ops, real.x, 0, global_log_tables());
    real.y = apply_chain_rt(p.ops, real.y, 0, global_log_tables());
  }
  const float2 y = __fmul2_rn(real, inv);
  const float2 t = __fadd2_rn(y, magic);
  const float2 f = __ffma2_rn(__fadd2_rn(t, make_float2(-kMagic, -kMagic)), make_float2(-1.0f, -1.0f), y);
  const float2 yy = __fmul2_rn(y, __fmul2_rn(y, make_float2(0x1p-31f, 0x1p-31f)));
  const float2 lhs = __ffma2_rn(f, f, yy);
  constexpr float kLim = 0.25f - 0x1p-15f - 0x1p-24f;  // exact in f32
  ok0 = lhs.x < kLim;
  ok1 = lhs.y < kLim;
  q0 = min(max((__float_as_int(t.x) - kMagicBits) + zo0, smin), smax);
  q1 = min(max((__float_as_int(t.y) - kMagicBits) + zo1, smin), smax);
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int m) {
  return m == 0 ? v.x : (m == 1 ? v.y : (m == 2 ? v.z : v.w));
}

// Four 16-byte row chunks (tile rows r0 + 32k, k = 0..3; local columns 16c .. 16c+15) -> their output
// codes, in place. Column parameters are loaded once for the four rows, row parameters once per row.
template <int QIN, int QOUT, bool OPS>
__device__ __forceinline__ void quant_rows(uint4 (&v)[4], int r0, int c, const QuantTilePlan& p, const QuantSmem& q) {
  float rs[4], ri[4];
  int rzm[4], rzo[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int row = r0 + 32 * k;
    rs[k] = QIN == 0 ? q.sin_[row] : p.qin.scale;
    rzm[k] = QIN == 0 ? q.zinm[row] : kMagicBits - p.qin.zp;
    ri[k] = QOUT == 0 ? q.inv[row] : p.qout.inv_scale;
    rzo[k] = QOUT == 0 ? q.zout[row] : p.qout.zp;
  }
  const int smin = p.qout.smin, smax = p.qout.smax;
  uint32_t o[4][4];
  uint32_t redo[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    int r[4][4];
#pragma unroll
    for (int b = 0; b < 4; b += 2) {
      const int jl = 16 * c + 4 * m + b;
      float2 cs = make_float2(0.f, 0.f), ci = make_float2(0.f, 0.f);
      int czm0 = 0, czm1 = 0, czo0 = 0, czo1 = 0;
      if (QIN == 1) {
        cs = *reinterpret_cast<const float2*>(&q.sin_[jl]);
        czm0 = q.zinm[jl];
        czm1 = q.zinm[jl + 1];
      }
      if (QOUT == 1) {
        ci = *reinterpret_cast<const float2*>(&q.inv[jl]);
        czo0 = q.zout[jl];
        czo1 = q.zout[jl + 1];
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t w = word_of(v[k], m);
        const int c0 = (int)(int8_t)(w >> (8 * b)), c1 = (int)(int8_t)(w >> (8 * b + 8));
        const float2 s2 = QIN == 1 ? cs : make_float2(rs[k], rs[k]);
        const float2 i2 = QOUT == 1 ? ci : make_float2(ri[k], ri[k]);
        bool ok0, ok1;
        quant_two<OPS>(c0, c1, s2, QIN == 1 ? czm0 : rzm[k], QIN == 1 ? czm1 : rzm[k], i2,
                       QOUT == 1 ? czo0 : rzo[k], QOUT == 1 ? czo1 : rzo[k], smin, smax, p, r[k][b], r[k][b + 1],
                       ok0, ok1);
        redo[k] |= ((ok0 ? 0u : 1u) | (ok1 ? 0u : 2u)) << (4 * m + b);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
      o[k][m] = __byte_perm(__byte_perm(r[k][0], r[k][1], 0x0040), __byte_perm(r[k][2], r[k][3], 0x0040), 0x5410);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t rk = redo[k];
    const int row = r0 + 32 * k;
#pragma unroll 1
    while (rk) {  // rare: the exact definition decides
      const int e = __ffs(rk) - 1;
      rk &= rk - 1;
      const int m = e >> 2, b = e & 3, jl = 16 * c + e;
      const int code = (int)(int8_t)(word_of(v[k], m) >> (8 * b));
      float sin, sout, inv;
      int zin, zout;
      quant_params<QIN, QOUT, OPS>(row, jl, p, q, sin, zin, sout, inv, zout);
      float real = dequant(code, sin, zin);
      if (OPS) real = apply_chain_rt(p.ops, real, 0, global_log_tables());
      const int res = quant_code_exact(real, sout, zout, smin, smax);
#pragma unroll
      for (int mm = 0; mm < 4; ++mm)  // static indices keep o in registers
        if (mm == m) o[k][mm] = (o[k][mm] & ~(0xFFu << (8 * b))) | (((uint32_t)res & 0xFFu) << (8 * b));
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) v[k] = make_uint4(o[k][0], o[k][1], o[k][2], o[k][3]);
}

// Dequantize -> quantize of four 16-byte row chunks without a float chain, for finite parameters with
// |scale_in / scale_out| < 2^13 (so |y| < 2^21 below). Per code:
//  * d = code - zp exactly: after flipping the sign bits, the byte (code + 128) becomes the low byte of
//    the f32 1.5*2^23, and subtracting 1.5*2^23 + 128 + zp is exact;
//  * real = RN(scale_in * d), as the definition has it; y = RN(real * RN(1/scale_out)) lies within
//    1.5*2^-23 (1 + 2^-22) |y| of the IEEE quotient RN(real / scale_out), so y(1 - 2^-22) and
//    y(1 + 2^-22) bracket it;
//  * t± = RN(y(1 ± 2^-22) + M) with M = 1.5*2^23 + zp_out (one FMA each) is M + the nearest integer to
//    y(1 ± 2^-22). When t+ = t-, no half-integer lies in the bracket (an end can be one only for
//    |y| >= 2^21, where the clamp decides anyway), so rint(quotient) + zp_out = bits(t) - bits(1.5*2^23).
// cvt.pack.sat saturates to [-128, 127]; CLAMP adds a narrower storage range. Words holding a code whose
// bracket contained a half-integer (about 1 in 10^4 at |y| ~ 100) are redone with the exact definition.
template <int QIN, int QOUT, bool CLAMP>
__device__ __forceinline__ void quant_rows_bracket(uint4 (&v)[4], int r0, int c, const QuantTilePlan& p,
                                                   const QuantSmem& q) {
  float rs[4], rz[4], ri[4], rm[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int row = r0 + 32 * k;
    rs[k] = QIN == 0 ? q.sin_[row] : p.qin.scale;
    rz[k] = QIN == 0 ? q.nzin[row] : -(kMagic + 128.0f + (float)p.qin.zp);
    ri[k] = QOUT == 0 ? q.inv[row] : p.qout.inv_scale;
    rm[k] = QOUT == 0 ? q.mout[row] : kMagic + (float)p.qout.zp;
  }
  const int smin = p.qout.smin, smax = p.qout.smax;
  const float2 kp = make_float2(1.0f + 0x1p-22f, 1.0f + 0x1p-22f), km = make_float2(1.0f - 0x1p-22f, 1.0f - 0x1p-22f);
  uint32_t o[4][4];
  uint32_t redo = 0u;  // bit 4k + m: word m of chunk k
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    uint32_t hi[4], dw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int b = 2; b >= 0; b -= 2) {  // codes 2, 3 first: their pack is the upper half of the word
      const int jl = 16 * c + 4 * m + b;
      float2 cs = make_float2(0.f, 0.f), cz = cs, ci = cs, cm = cs;
      if (QIN == 1) {
        cs = *reinterpret_cast<const float2*>(&q.sin_[jl]);
        cz = *reinterpret_cast<const float2*>(&q.nzin[jl]);
      }
      if (QOUT == 1) {
        ci = *reinterpret_cast<const float2*>(&q.inv[jl]);
        cm = *reinterpret_cast<const float2*>(&q.mout[jl]);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t w = word_of(v[k], m) ^ 0x80808080u;
        const float2 e = make_float2(__uint_as_float(__byte_perm(w, (uint32_t)kMagicBits, 0x7650u | b)),
                                     __uint_as_float(__byte_perm(w, (uint32_t)kMagicBits, 0x7650u | (b + 1))));
        const float2 df = __fadd2_rn(e, QIN == 1 ? cz : make_float2(rz[k], rz[k]));
        const float2 real = __fmul2_rn(QIN == 1 ? cs : make_float2(rs[k], rs[k]), df);
        const float2 y = __fmul2_rn(real, QOUT == 1 ? ci : make_float2(ri[k], ri[k]));
        const float2 mm = QOUT == 1 ? cm : make_float2(rm[k], rm[k]);
        const float2 tp = __ffma2_rn(y, kp, mm), tm = __ffma2_rn(y, km, mm);
        dw[k] |= (__float_as_uint(tp.x) ^ __float_as_uint(tm.x)) | (__float_as_uint(tp.y) ^ __float_as_uint(tm.y));
        int q0 = __float_as_int(tp.x) - kMagicBits, q1 = __float_as_int(tp.y) - kMagicBits;
        if (CLAMP) {
          q0 = min(max(q0, smin), smax);
          q1 = min(max(q1, smin), smax);
        }
        if (b == 2) asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, 0;" : "=r"(hi[k]) : "r"(q1), "r"(q0));
        else asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(o[k][m]) : "r"(q1), "r"(q0), "r"(hi[k]));
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) redo |= (dw[k] != 0u ? 1u : 0u) << (4 * k + m);
  }
#pragma unroll 1
  while (redo) {  // rare: the exact definition decides the word's four codes
    const int e = __ffs(redo) - 1;
    redo &= redo - 1;
    const int k = e >> 2, m = e & 3, row = r0 + 32 * k;
    const uint32_t w = word_of(v[k], m);
    uint32_t res = 0u;
    for (int b = 0; b < 4; ++b) {
      float sin, sout, inv;
      int zin, zout;
      quant_params<QIN, QOUT, false>(row, 16 * c + 4 * m + b, p, q, sin, zin, sout, inv, zout);
      const int code = (int)(int8_t)(w >> (8 * b));
      res |= ((uint32_t)quant_code_exact(dequant(code, sin, zin), sout, zout, smin, smax) & 0xFFu) << (8 * b);
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)  // static indices keep o in registers
#pragma unroll
      for (int mm = 0; mm < 4; ++mm)
        if (kk == k && mm == m) o[kk][mm] = res;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) v[k] = make_uint4(o[k][0], o[k][1], o[k][2], o[k][3]);
}

template <int QIN, int QOUT, bool OPS>
__global__ void __launch_bounds__(256, 4) quant_tile_kernel(QuantTilePlan p, int64_t ntj) {
  __shared__ __align__(16) uint32_t tile[kQT * kQT / 4];  // 128 rows x 32 words, word column swizzled
  __shared__ QuantSmem q;
  const int t = threadIdx.x;
  const int64_t ti = blockIdx.x / ntj, tj = blockIdx.x % ntj;
  const int64_t i0 = ti * kQT, j0 = tj * kQT;
  const int64_t n0 = p.n0, n1 = p.n1;
  // stage the per-axis parameters of this tile
  bool bad = false;
  if (t < kQT) {
    const int64_t i = i0 + t, j = j0 + t;
    if (p.qin.axis == 0 && i < n0) { q.sin_[t] = p.qin.scales[i]; q.zin[t] = p.qin.zps[i]; }
    if (p.qin.axis == 1 && j < n1) { q.sin_[t] = p.qin.scales[j]; q.zin[t] = p.qin.zps[j]; }
    float a = fabsf(p.qin.scale), b = fabsf(p.qout.inv_scale);
    if (p.qin.axis >= 0 && (p.qin.axis == 0 ? i < n0 : j < n1)) {
      q.zinm[t] = kMagicBits - q.zin[t];
      q.nzin[t] = -(kMagic + 128.0f + (float)q.zin[t]);
      a = fabsf(q.sin_[t]);
    }
    const int64_t k = p.qout.axis == 0 ? i : j;
    if (p.qout.axis >= 0 && k < (p.qout.axis == 0 ? n0 : n1)) {
      const float s = p.qout.scales[k];
      q.sout[t] = s;
      q.inv[t] = __frcp_rn(s);
      q.zout[t] = p.qout.zps[k];
      q.mout[t] = kMagic + (float)q.zout[t];
      b = fabsf(q.inv[t]);
    }
    bad = !(a < 0x1p60f && b < 0x1p60f && a * b < 8192.0f);  // outside quant_rows_bracket's range
  }
  const int slow = __syncthreads_or(bad);
  const bool full = (i0 + kQT <= n0) && (j0 + kQT <= n1) && (n0 % 16 == 0) && (n1 % 16 == 0) &&
                    ((uintptr_t)p.in % 16 == 0) && ((uintptr_t)p.out % 16 == 0);
  if (!full) {
    quant_tile_ragged(p, i0, j0, reinterpret_cast<uint8_t*>(tile), q);
    return;
  }
  // 128 rows x 8 chunks of 16 bytes; chunk (row, c) stored at word column 4 * (c ^ ((row >> 4) & 7))
  uint4 v[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int qd = t + 256 * k, row = qd >> 3, c = qd & 7;
    const uint4* src = reinterpret_cast<const uint4*>(p.in + (i0 + row) * n1 + j0 + 16 * c);
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v[k].x), "=r"(v[k].y), "=r"(v[k].z), "=r"(v[k].w)
                 : "l"(src));
  }
  if (!OPS && !slow) {  // rows t/8 + 32k, chunk t%8
    if (p.qout.smin > -128 || p.qout.smax < 127) quant_rows_bracket<QIN, QOUT, true>(v, t >> 3, t & 7, p, q);
    else quant_rows_bracket<QIN, QOUT, false>(v, t >> 3, t & 7, p, q);
  } else {
    quant_rows<QIN, QOUT, OPS>(v, t >> 3, t & 7, p, q);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int qd = t + 256 * k, row = qd >> 3, c = qd & 7;
    const int wc = 4 * (c ^ ((row >> 4) & 7));
    *reinterpret_cast<uint4*>(&tile[row * 32 + wc]) = v[k];
  }
  __syncthreads();
  // unit: word column jg (output rows 4jg..4jg+3), 16-row chunk ic
  const int jg = t >> 3, ic = t & 7;
  uint32_t w[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) w[k] = tile[(16 * ic + k) * 32 + (jg ^ (4 * ic))];
  uint32_t outw[4][4];  // [q][m]
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t a = w[4 * m], b = w[4 * m + 1], c = w[4 * m + 2], d = w[4 * m + 3];
    const uint32_t t0 = __byte_perm(a, b, 0x5140), t1 = __byte_perm(a, b, 0x7362);
    const uint32_t t2 = __byte_perm(c, d, 0x5140), t3 = __byte_perm(c, d, 0x7362);
    outw[0][m] = __byte_perm(t0, t2, 0x5410);
    outw[1][m] = __byte_perm(t0, t2, 0x7632);
    outw[2][m] = __byte_perm(t1, t3, 0x5410);
    outw[3][m] = __byte_perm(t1, t3, 0x7632);
  }
#pragma unroll
  for (int qq = 0; qq < 4; ++qq) {
    uint4* dst = reinterpret_cast<uint4*>(p.out + (j0 + 4 * jg + qq) * n0 + i0 + 16 * ic);
    *dst = make_uint4(outw[qq][0], outw[qq][1], outw[qq][2], outw[qq][3]);
  }
}

template <int QIN, int QOUT>
static cudaError_t quant_launch2(const QuantTilePlan& p, int64_t blocks, int64_t ntj, cudaStream_t s) {
  if (p.ops.n) quant_tile_kernel<QIN, QOUT, true><<<(unsigned)blocks, 256, 0, s>>>(p, ntj);
  else quant_tile_kernel<QIN, QOUT, false><<<(unsigned)blocks, 256, 0, s>>>(p, ntj);
  return cudaGetLastError();
}

template <int QIN>
static cudaError_t quant_launch1(const QuantTilePlan& p, int64_t blocks, int64_t ntj, cudaStream_t s) {
  if (p.qout.axis == 0) return quant_launch2<QIN, 0>(p, blocks, ntj, s);
  if (p.qout.axis == 1) return quant_launch2<QIN, 1>(p, blocks, ntj, s);
  return quant_launch2<QIN, -1>(p, blocks, ntj, s);
}

// ---------------------------------------------------------------------------------------------
// Tensor-copy quantized relayout: whole 128 x 128 tiles (n0, n1 multiples of 128), 16-byte aligned
// buffers, no float chain, per-tensor output parameters.
//   * Tile (ti, tj) lands by one 2-D tensor copy with the 128-byte swizzle (16-byte chunk c of row r at
//     chunk c ^ (r % 8)); a per-axis input parameter slice (128 scales, 128 zero points) comes with it
//     by two 1-D bulk copies on the same mbarrier.
//   * Warp w converts chunk w (columns 16w .. 16w+15) of rows lane + 32k: the swizzle spreads a quarter
//     warp's eight rows over eight bank groups, and per-column parameters are the same for the whole
//     warp (broadcast reads).
//   * The codes go to an output tile with chunk c of row r at c ^ ((r ^ (r / 16)) % 8): conflict-free for
//     those writes (8 consecutive rows) and for the transposed reads (16 rows of one word column, 8
//     sixteen-row groups per instruction), then 4x4 byte transposes and 16-byte stores as in
//     quant_tile_kernel.
//   * After its stores each warp counts itself done with the stage; the last one refills it with the
//     block's tile j + kQStages. A second barrier per tile frees the output tile.
// The arithmetic is quant_rows_bracket's (see there), with the exact definition for bracketed ties and
// for tiles whose parameters fall outside the bracket's range.
// ---------------------------------------------------------------------------------------------
constexpr int kQStages = 2;
constexpr int kQWarps = 8;
struct QTmaShared {
  float ps[kQStages][kQT];    // per-axis input scales of the stage's tile
  int32_t pz[kQStages][kQT];  // and zero points
  int2 tile[kQStages];        // (ti, tj) of the stage's tile
  int done[kQStages];         // warps done with the stage's tile
  uint64_t full[kQStages];
};

static size_t quant_tma_smem_bytes() {
  return 1024 /* alignment slack */ + (size_t)(kQStages + 1) * kQT * kQT + sizeof(QTmaShared);
}

template <int QIN, bool CLAMP>
__global__ void __launch_bounds__(256, 4)
    quant_tma_kernel(const __grid_constant__ CUtensorMap tmap, QuantTilePlan p, int64_t ntj, int64_t n_tiles) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint32_t* otile = reinterpret_cast<uint32_t*>(base + kQStages * kQT * kQT);  // 128 rows x 32 words
  QTmaShared& qs = *reinterpret_cast<QTmaShared*>(otile + kQT * kQT / 4);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  auto issue = [&](int64_t it, int64_t j) {
    const int st = (int)(j % kQStages);
    const int64_t ti = it / ntj, tj = it % ntj;
    qs.tile[st] = make_int2((int)ti, (int)tj);
    const uint32_t bar = smem_addr(&qs.full[st]);
    mbar_arrive_expect_tx(bar, kQT * kQT + (QIN >= 0 ? 2u * kQT * 4u : 0u));
    tma_load_2d(base + st * kQT * kQT, &tmap, (int32_t)(tj * kQT), (int32_t)(ti * kQT), bar);
    if (QIN >= 0) {
      const int64_t k0 = (QIN == 0 ? ti : tj) * kQT;
      bulk_load(qs.ps[st], p.qin.scales + k0, kQT * 4, bar);
      bulk_load(qs.pz[st], p.qin.zps + k0, kQT * 4, bar);
    }
  };
  if (tid == 0) {
    prefetch_tensor_map(&tmap);
    for (int st = 0; st < kQStages; ++st) {
      mbar_init(smem_addr(&qs.full[st]), 1);
      qs.done[st] = 0;
    }
    fence_mbar_init();
    for (int64_t j = 0; j < kQStages; ++j) {
      const int64_t it = blockIdx.x + j * gridDim.x;
      if (it < n_tiles) issue(it, j);
    }
  }
  __syncthreads();
  const int64_t n0 = p.n0;
  const float so = p.qout.scale, io = p.qout.inv_scale;
  const int zo = p.qout.zp, smin = p.qout.smin, smax = p.qout.smax;
  const float mo = kMagic + (float)zo;
  // The product of the input scale and RN(1/scale_out) is formed once per parameter, so y = RN(d * P),
  // d = code - z: P is within 2^-24 of s * RN(1/s_out), which is within 2^-24 of s / s_out, and the
  // product and RN(s d) (the dequantized value) round once more each, so y lies within 4 * 2^-24 (plus
  // second-order terms) of RN(s d) / s_out and 5 * 2^-24 of the IEEE quotient rounded: the bracket
  // y(1 +- 2^-21) holds it with room.
  const float2 kp = make_float2(1.0f + 0x1p-21f, 1.0f + 0x1p-21f), km = make_float2(1.0f - 0x1p-21f, 1.0f - 0x1p-21f);
  int64_t j = 0;
  for (int64_t item = blockIdx.x; item < n_tiles; item += gridDim.x, ++j) {
    const int st = (int)(j % kQStages);
    const bool arrived = mbar_wait(smem_addr(&qs.full[st]), (uint32_t)((j / kQStages) & 1));
    const int2 tt = qs.tile[st];
    const uint8_t* rt = base + st * kQT * kQT;
    const float* ps = qs.ps[st];
    const int32_t* pz = qs.pz[st];
    // this thread's codes: chunk w of rows lane + 32k (the tensor copy's swizzle: chunk c at c ^ (r % 8))
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = lane + 32 * k;
      v[k] = *reinterpret_cast<const uint4*>(rt + r * kQT + 16 * (w ^ (r & 7)));
    }
    // parameters: per row (QIN 0), per column (QIN 1, the same for the whole warp) or per tensor. With
    // the zero point z, -(1.5*2^23 + 128 + z) has the bits of 1.5*2^23 plus 128 + z (in [0, 255]) and the
    // sign bit: df = e + that = code - z exactly.
    float rs[4], rz[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int zz = QIN == 0 ? pz[lane + 32 * k] : p.qin.zp;
      rs[k] = QIN == 0 ? ps[lane + 32 * k] : p.qin.scale;
      rz[k] = __int_as_float((kMagicBits + 128 + zz) | (int)0x80000000u);
    }
    float rp[4];  // per row (or tensor): scale * RN(1/scale_out)
#pragma unroll
    for (int k = 0; k < 4; ++k) rp[k] = __fmul_rn(rs[k], io);
    // the bracket needs finite parameters with |scale_in / scale_out| < 2^13: known from the host copies
    // when they were given, else checked on this thread's parameters
    bool bad;
    if (p.qin.max_abs_scale >= 0.0f) {
      bad = !(fabsf(io) < 0x1p60f && p.qin.max_abs_scale < 0x1p60f && p.qin.max_abs_scale * fabsf(io) < 8192.0f);
    } else {
      bad = !(fabsf(io) < 0x1p60f);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (QIN != 1) bad |= !(fabsf(rs[k]) < 0x1p60f && fabsf(rs[k]) * fabsf(io) < 8192.0f);
      if (QIN == 1) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float sc = ps[16 * w + c];
          bad |= !(fabsf(sc) < 0x1p60f && fabsf(sc) * fabsf(io) < 8192.0f);
        }
      }
    }
    uint32_t o[4][4];
    if (!bad) {
      uint32_t redo = 0u;  // bit 4k + m: word m of row k
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        uint32_t hi[4], dw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int b = 2; b >= 0; b -= 2) {  // codes 2, 3 first: their pack is the upper half of the word
          float2 cp = make_float2(0.f, 0.f), cz = cp;
          if (QIN == 1) {
            const int jl = 16 * w + 4 * m + b;
            cp = __fmul2_rn(*reinterpret_cast<const float2*>(&ps[jl]), make_float2(io, io));
            const int2 zz = *reinterpret_cast<const int2*>(&pz[jl]);
            cz = make_float2(__int_as_float((kMagicBits + 128 + zz.x) | (int)0x80000000u),
                             __int_as_float((kMagicBits + 128 + zz.y) | (int)0x80000000u));
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t wd = word_of(v[k], m) ^ 0x80808080u;
            const float2 e = make_float2(__uint_as_float(__byte_perm(wd, (uint32_t)kMagicBits, 0x7650u | b)),
                                         __uint_as_float(__byte_perm(wd, (uint32_t)kMagicBits, 0x7650u | (b + 1))));
            const float2 df = __fadd2_rn(e, QIN == 1 ? cz : make_float2(rz[k], rz[k]));
            const float2 y = __fmul2_rn(QIN == 1 ? cp : make_float2(rp[k], rp[k]), df);
            const float2 tp = __ffma2_rn(y, kp, make_float2(mo, mo)), tm = __ffma2_rn(y, km, make_float2(mo, mo));
            dw[k] |= (__float_as_uint(tp.x) ^ __float_as_uint(tm.x)) | (__float_as_uint(tp.y) ^ __float_as_uint(tm.y));
            int q0 = __float_as_int(tp.x) - kMagicBits, q1 = __float_as_int(tp.y) - kMagicBits;
            if (CLAMP) {
              q0 = min(max(q0, smin), smax);
              q1 = min(max(q1, smin), smax);
            }
            if (b == 2) asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, 0;" : "=r"(hi[k]) : "r"(q1), "r"(q0));
            else asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(o[k][m]) : "r"(q1), "r"(q0), "r"(hi[k]));
          }
        }
        if (dw[0] | dw[1] | dw[2] | dw[3]) {  // rare: mark the words with an undecided code
#pragma unroll
          for (int k = 0; k < 4; ++k) redo |= (dw[k] != 0u ? 1u : 0u) << (4 * k + m);
        }
      }
#pragma unroll 1
      while (redo) {  // rare: the exact definition decides the word's four codes
        const int e = __ffs(redo) - 1;
        redo &= redo - 1;
        const int k = e >> 2, m = e & 3, r = lane + 32 * k;
        const uint32_t wd = word_of(v[k], m);
        uint32_t res = 0u;
        for (int b = 0; b < 4; ++b) {
          const int jl = 16 * w + 4 * m + b;
          const float sin = QIN == 0 ? ps[r] : QIN == 1 ? ps[jl] : p.qin.scale;
          const int zin = QIN == 0 ? pz[r] : QIN == 1 ? pz[jl] : p.qin.zp;
          const int code = (int)(int8_t)(wd >> (8 * b));
          res |= ((uint32_t)quant_code_exact(dequant(code, sin, zin), so, zo, smin, smax) & 0xFFu) << (8 * b);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // static indices keep o in registers
#pragma unroll
          for (int mm = 0; mm < 4; ++mm)
            if (kk == k && mm == m) o[kk][mm] = res;
      }
    } else {
      // parameters outside the bracket's range (or not finite): the exact definition for every code
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int r = lane + 32 * k;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const uint32_t wd = word_of(v[k], m);
          uint32_t res = 0u;
#pragma unroll 1
          for (int b = 0; b < 4; ++b) {
            const int jl = 16 * w + 4 * m + b;
            const float sin = QIN == 0 ? ps[r] : QIN == 1 ? ps[jl] : p.qin.scale;
            const int zin = QIN == 0 ? pz[r] : QIN == 1 ? pz[jl] : p.qin.zp;
            const int code = (int)(int8_t)(wd >> (8 * b));
            res |= ((uint32_t)quant_code_exact(dequant(code, sin, zin), so, zo, smin, smax) & 0xFFu) << (8 * b);
          }
          o[k][m] = res;
        }
      }
    }
    // output tile: chunk w of row r at chunk w ^ ((r ^ (r / 16)) % 8)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = lane + 32 * k;
      *reinterpret_cast<uint4*>(&otile[r * 32 + 4 * (w ^ ((r ^ (r >> 4)) & 7))]) =
          make_uint4(o[k][0], o[k][1], o[k][2], o[k][3]);
    }
    if (__syncthreads_or(arrived ? 0 : 1)) {
      // a copy did not arrive in time: record the fault, wait (bounded) for this block's copies still
      // in flight, leave the rest of its outputs unwritten and return
      if (tid == 0) {
        record_fault(kFaultCopyTimeout);
        for (int64_t q = j; q < j + kQStages && blockIdx.x + q * gridDim.x < n_tiles; ++q)
          mbar_wait(smem_addr(&qs.full[q % kQStages]), (uint32_t)((q / kQStages) & 1));
      }
      return;
    }
    // the stage has been read by every warp (its codes are in the output tile): the last warp out refills it
    if (lane == 0) {
      __threadfence_block();
      if (atomicAdd(&qs.done[st], 1) == kQWarps - 1) {
        qs.done[st] = 0;
        const int64_t nxt = item + (int64_t)kQStages * gridDim.x;
        if (nxt < n_tiles) {
          fence_proxy_async();
          issue(nxt, j + kQStages);
        }
      }
    }
    // transposed: word column jg (output rows 4jg..4jg+3), sixteen-row group ic
    const int jg = tid >> 3, ic = tid & 7;
    uint32_t wv[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) wv[k] = otile[(16 * ic + k) * 32 + 4 * ((jg >> 2) ^ ((k ^ ic) & 7)) + (jg & 3)];
    uint32_t outw[4][4];  // [q][m]
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint32_t a = wv[4 * m], b = wv[4 * m + 1], c = wv[4 * m + 2], d = wv[4 * m + 3];
      const uint32_t t0 = __byte_perm(a, b, 0x5140), t1 = __byte_perm(a, b, 0x7362);
      const uint32_t t2 = __byte_perm(c, d, 0x5140), t3 = __byte_perm(c, d, 0x7362);
      outw[0][m] = __byte_perm(t0, t2, 0x5410);
      outw[1][m] = __byte_perm(t0, t2, 0x7632);
      outw[2][m] = __byte_perm(t1, t3, 0x5410);
      outw[3][m] = __byte_perm(t1, t3, 0x7632);
    }
    const int64_t i0 = (int64_t)tt.x * kQT, j0 = (int64_t)tt.y * kQT;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      uint4* dst = reinterpret_cast<uint4*>(p.out + (j0 + 4 * jg + qq) * n0 + i0 + 16 * ic);
      *dst = make_uint4(outw[qq][0], outw[qq][1], outw[qq][2], outw[qq][3]);
    }
    __syncthreads();  // the output tile is rewritten by the next tile
  }
}

// An s8 tensor map over the [n0, n1] row-major input with 128 x 128 boxes and the 128-byte swizzle;
// false if it cannot be made.
static bool make_quant_tensor_map(const QuantTilePlan& p, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)p.n1, (cuuint64_t)p.n0};
  const cuuint64_t strides[1] = {(cuuint64_t)p.n1};
  const cuuint32_t box[2] = {kQT, kQT};
  const cuuint32_t elem_strides[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(p.in), dims, strides, box, elem_strides,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int QIN>
static cudaError_t quant_tma_launch(const QuantTilePlan& p, const CUtensorMap& map, int64_t n_tiles, int64_t ntj,
                                    cudaStream_t s) {
  const bool clamp = p.qout.smin > -128 || p.qout.smax < 127;
  const void* kernel = clamp ? (const void*)quant_tma_kernel<QIN, true> : (const void*)quant_tma_kernel<QIN, false>;
  const size_t smem = quant_tma_smem_bytes();
  const int nb = kernel_blocks_per_sm(kernel, 256, smem);
  // one wave of every resident block: tiles dealt round-robin, the first kQStages of each block's
  // requested at once
  int64_t grid = (int64_t)device_sm_count() * nb;
  if (grid > n_tiles) grid = n_tiles;
  if (grid < 1) grid = 1;
  if (clamp) quant_tma_kernel<QIN, true><<<(unsigned)grid, 256, smem, s>>>(map, p, ntj, n_tiles);
  else quant_tma_kernel<QIN, false><<<(unsigned)grid, 256, smem, s>>>(map, p, ntj, n_tiles);
  return cudaGetLastError();
}

cudaError_t launch_quant_tile(const QuantTilePlan& p, cudaStream_t s) {
  const int64_t nti = (p.n0 + kQT - 1) / kQT, ntj = (p.n1 + kQT - 1) / kQT;
  const int64_t blocks = nti * ntj;
  if (blocks == 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  // whole tiles, aligned buffers and parameters, no float chain, per-tensor output: tensor copies
  const bool tma_shape = p.n0 % kQT == 0 && p.n1 % kQT == 0 && p.ops.n == 0 && p.qout.axis < 0 &&
                         (uintptr_t)p.in % 16 == 0 && (uintptr_t)p.out % 16 == 0 && nti <= 0x7FFFFFFF &&
                         ntj <= 0x7FFFFFFF &&
                         (p.qin.axis < 0 || ((uintptr_t)p.qin.scales % 16 == 0 && (uintptr_t)p.qin.zps % 16 == 0));
  CUtensorMap map;
  if (tma_shape && make_quant_tensor_map(p, &map)) {
    if (p.qin.axis == 0) return quant_tma_launch<0>(p, map, blocks, ntj, s);
    if (p.qin.axis == 1) return quant_tma_launch<1>(p, map, blocks, ntj, s);
    return quant_tma_launch<-1>(p, map, blocks, ntj, s);
  }
  if (p.qin.axis == 0) return quant_launch1<0>(p, blocks, ntj, s);
  if (p.qin.axis == 1) return quant_launch1<1>(p, blocks, ntj, s);
  return quant_launch1<-1>(p, blocks, ntj, s);
}

}  // namespace hlo
