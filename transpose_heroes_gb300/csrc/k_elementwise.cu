// Elementwise kernel for fusions whose transpose is the identity on memory (same physical order in and
// out): the loop emitter of "XLA:GPU Emitters" (section "Loop emitter": a linear walk over the output
// so that writes are coalesced, with vectorized loads and stores, section "Vectorization").
#include <cooperative_groups.h>

#include <map>
#include <mutex>

#include "device_common.cuh"

namespace hlo {
#include "tanh_table.inc"  // kTanhBf16: tanh rounded to bf16 for every bf16 |x|
}  // namespace hlo

namespace cg = cooperative_groups;

namespace hlo {

struct EwPlan {
  const void* in;
  void* out;
  int64_t n;
  int dt;
  Chain pro, epi;
};

__device__ __forceinline__ float ew_apply(const EwPlan& p, float v, const LogTab& lt) {
  v = apply_chain_rt(p.pro, v, 0, lt);
  return apply_chain_rt(p.epi, v, 0, lt);
}

// Two elements of log through the first pass, the rest of the correctly rounded log where it
// leaves the rounding open (same result as cr_logf).
__device__ __forceinline__ void log2x(float& a, float& b, const float* l1i, const float* l1h, const float* l1l,
                                      const LogTab& lt) {
  float ya, yb;
  bool oa, ob;
  cr_logf_first2(a, b, l1i, l1h, l1l, ya, yb, oa, ob);
  a = oa ? ya : cr_logf(a, lt.c, lt.e);
  b = ob ? yb : cr_logf(b, lt.c, lt.e);
}

template <bool VEC>
__global__ void __launch_bounds__(256) elementwise_f32_kernel(EwPlan p) {
  __shared__ float4 s_lc[HLO_LOG_NC];
  __shared__ float2 s_le[HLO_LOG_NE];
  __shared__ float s_l1[3][32];
  load_log_tables(s_lc, s_le);
  load_log1_tables(s_l1[0], s_l1[1], s_l1[2]);
  __syncthreads();
  const LogTab lt = {s_lc, s_le};
  const bool pure_log = p.pro.n == 1 && p.pro.op[0] == OP_LOG && p.epi.n == 0;
  const float* in = reinterpret_cast<const float*>(p.in);
  float* out = reinterpret_cast<float*>(p.out);
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t done = 0;
  if (VEC) {
    const int64_t nv = p.n / 4;
    for (int64_t v = tid; v < nv; v += stride) {
      float4 x = __ldg(reinterpret_cast<const float4*>(in) + v);
      if (pure_log) {
        log2x(x.x, x.y, s_l1[0], s_l1[1], s_l1[2], lt);
        log2x(x.z, x.w, s_l1[0], s_l1[1], s_l1[2], lt);
      } else {
        x.x = ew_apply(p, x.x, lt);
        x.y = ew_apply(p, x.y, lt);
        x.z = ew_apply(p, x.z, lt);
        x.w = ew_apply(p, x.w, lt);
      }
      reinterpret_cast<float4*>(out)[v] = x;
    }
    done = nv * 4;
  }
  for (int64_t e = done + tid; e < p.n; e += stride) out[e] = ew_apply(p, in[e], lt);
}

__global__ void __launch_bounds__(256) elementwise_any_kernel(EwPlan p) {
  const LogTab lt = global_log_tables();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < p.n; e += stride) {
    float v = ew_apply(p, load_as_f32(p.in, p.dt, e), lt);
    store_from_f32(p.out, p.dt, e, round_to_dt(v, p.dt));
  }
}

// ---- 16-bit float chains, every op rounded to the element type ----------------------------------
// Eight elements per 16-byte vector, held as four packed pairs. Adds and multiplies (by the input or
// by a constant) run as packed bf16x2 / f16x2 instructions, which round each lane's exact result once:
// the spec's per-op semantics. exp, log and tanh unpack a pair to f32 and use the correctly rounded
// 16-bit versions. The ops are walked once per vector, so their dispatch is shared by eight elements.
template <int DT>
__device__ __forceinline__ uint32_t pk_add(uint32_t a, uint32_t b) {
  uint32_t r;
  if (DT == BF16) asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  else asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

template <int DT>
__device__ __forceinline__ uint32_t pk_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  if (DT == BF16) asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  else asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

template <int DT>
__device__ __forceinline__ float pk_lo(uint32_t w) {
  return DT == BF16 ? __uint_as_float(w << 16) : f16_bits_to_f32((uint16_t)(w & 0xFFFFu));
}

template <int DT>
__device__ __forceinline__ float pk_hi(uint32_t w) {
  return DT == BF16 ? __uint_as_float(w & 0xFFFF0000u) : f16_bits_to_f32((uint16_t)(w >> 16));
}

// Two f32 values that are already values of the 16-bit type, packed (exactly).
template <int DT>
__device__ __forceinline__ uint32_t pk_pack(float lo, float hi) {
  uint32_t r;
  if (DT == BF16) asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  else asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

template <int DT>
__device__ __forceinline__ uint32_t pk_splat(float c) {
  const uint32_t b = DT == BF16 ? (__float_as_uint(c) >> 16) : (uint32_t)f32_to_f16_bits(c);
  return b | (b << 16);
}

// tanh in f32 for the bf16 path, two lanes per f32x2 instruction, within 16 f32 ulps of tanh(x) for
// every bf16 x (checked over all of them): |x| < 0.55: x P(x^2), P a degree-5 fit of tanh(x)/x;
// otherwise (1 - e)/(1 + e), e = e^{-2|x|} from the SFU exponential and reciprocal.
__device__ __forceinline__ float2 tanh_fast2(float2 x) {
  const float2 ax = make_float2(fabsf(x.x), fabsf(x.y));
  const float2 s = __fmul2_rn(x, x);
  float2 p = __ffma2_rn(s, make_float2(-0.006230350583791733f, -0.006230350583791733f),
                        make_float2(0.02103571780025959f, 0.02103571780025959f));
  p = __ffma2_rn(p, s, make_float2(-0.05384165421128273f, -0.05384165421128273f));
  p = __ffma2_rn(p, s, make_float2(0.1333244889974594f, 0.1333244889974594f));
  p = __ffma2_rn(p, s, make_float2(-0.3333331048488617f, -0.3333331048488617f));
  p = __ffma2_rn(p, s, make_float2(1.0f, 1.0f));
  const float2 small = __fmul2_rn(x, p);
  const float2 t = __fmul2_rn(ax, make_float2(-2.885390081777927f, -2.885390081777927f));
  float2 e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.x) : "f"(t.x));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.y) : "f"(t.y));
  const float2 d = __fadd2_rn(e, make_float2(1.0f, 1.0f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.x) : "f"(d.x));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.y) : "f"(d.y));
  const float2 big = __fmul2_rn(__ffma2_rn(e, make_float2(-1.0f, -1.0f), make_float2(1.0f, 1.0f)), r);
  return make_float2(ax.x < 0.55f ? small.x : copysignf(big.x, x.x), ax.y < 0.55f ? small.y : copysignf(big.y, x.y));
}

// True when every f32 value within `ulps` ulps of y rounds to bf16 the way y does: the 16 bits bf16
// drops are not within `ulps` of the midpoint 0x8000 (ulps are uniform inside a binade and through
// the subnormals; inf and NaN pass).
__device__ __forceinline__ bool bf16_clear_of_midpoint(float y, int ulps) {
  const uint32_t b = __float_as_uint(y);
  const int d = (int)(b & 0xFFFFu) - 0x8000;
  return (d > ulps || d < -ulps) || ((b & 0x7F800000u) == 0x7F800000u);
}

// exp, log or tanh of one packed pair, correctly rounded to the 16-bit type, the slow way (the
// correctly rounded per-element path); out of line, as the fast path below rarely needs it.
template <int DT>
static __device__ __noinline__ uint32_t fn2_exact(int op, uint32_t w, const LogTab& lt) {
  return pk_pack<DT>(apply_op(op, pk_lo<DT>(w), 0.f, 0.f, 0.f, true, DT, lt),
                     apply_op(op, pk_hi<DT>(w), 0.f, 0.f, 0.f, true, DT, lt));
}

// exp, log or tanh of one packed bf16 pair from an f32 approximation: returns false (and leaves w
// unchanged) when a lane's f32 value lies too close to a bf16 rounding midpoint to decide it.
template <int OP>
__device__ __forceinline__ bool bf16_fn2_fast(uint32_t& w, const LogTab& lt) {
  const float a = pk_lo<BF16>(w), b = pk_hi<BF16>(w);
  float2 f;
  int ulps = 2;  // expf is within 2 ulps; cr_logf is correctly rounded
  if (OP == OP_TANH) {
    f = tanh_fast2(make_float2(a, b));
    ulps = 16;
  } else if (OP == OP_EXP) {
    f = make_float2(expf(a), expf(b));
  } else {
    f = make_float2(cr_logf(a, lt.c, lt.e), cr_logf(b, lt.c, lt.e));
  }
  // the f32 value's bf16 rounding is the correct one unless the bits it drops lie within `ulps`
  // of the midpoint
  if (!(bf16_clear_of_midpoint(f.x, ulps) & bf16_clear_of_midpoint(f.y, ulps))) return false;
  w = pk_pack<BF16>(f.x, f.y);
  return true;
}

// One transcendental op on kV packed pairs: the fast path for every pair, then the exact path for
// the pairs it could not decide (one branch per op, not per pair).
template <int DT, int OP, int kV>
__device__ __forceinline__ void fn16x2(uint32_t (&v)[kV], const LogTab& lt) {
  if (DT == BF16) {
    uint32_t open = 0u;
#pragma unroll
    for (int j = 0; j < kV; ++j) open |= (bf16_fn2_fast<OP>(v[j], lt) ? 0u : 1u) << j;
    if (open) {
#pragma unroll
      for (int j = 0; j < kV; ++j)
        if (open & (1u << j)) v[j] = fn2_exact<DT>(OP, v[j], lt);
    }
  } else {
#pragma unroll
    for (int j = 0; j < kV; ++j) v[j] = fn2_exact<DT>(OP, v[j], lt);
  }
}

// One pair through exp, log or tanh: the fast path, then the exact one if needed, in one out-of-line
// call (the streaming kernel keeps its registers for the data).
template <int DT>
static __device__ __noinline__ uint32_t fn2_call(int op, uint32_t w, const LogTab& lt) {
  if (DT == BF16) {
    uint32_t r = w;
    const bool ok = op == OP_TANH  ? bf16_fn2_fast<OP_TANH>(r, lt)
                    : op == OP_EXP ? bf16_fn2_fast<OP_EXP>(r, lt)
                                   : bf16_fn2_fast<OP_LOG>(r, lt);
    if (ok) return r;
  }
  return fn2_exact<DT>(op, w, lt);
}

// tanh of a packed bf16 pair from the table of kTanhBf16 (in shared memory): the entry of |x|, with
// the sign of x.
__device__ __forceinline__ uint32_t tanh_bf16x2_tab(uint32_t w, const uint16_t* tab) {
  const uint32_t a = w & 0x7FFF7FFFu;
  const uint32_t lo = tab[a & 0xFFFFu], hi = tab[a >> 16];
  return __byte_perm(lo, hi, 0x5410) | (w & 0x80008000u);
}

// The chain on kV packed pairs (2 kV elements); the op dispatch is shared by all of them. With TT,
// bf16 tanh reads the table at `ttab` and the chain has no exp or log (the caller makes sure: their
// code would take registers from the data); with OOL, exp, log (and tanh without the table) run out
// of line.
template <int DT, int kV, bool TT = false, bool OOL = false>
__device__ __forceinline__ void chain16x2(const Chain& c, uint32_t (&v)[kV], const uint32_t (&x)[kV], const LogTab& lt,
                                          const uint16_t* ttab = nullptr) {
#pragma unroll 1
  for (int k = 0; k < c.n; ++k) {
    switch (c.op[k]) {
      case OP_MUL_IN:
#pragma unroll
        for (int j = 0; j < kV; ++j) v[j] = pk_mul<DT>(v[j], x[j]);
        break;
      case OP_ADD_IN:
#pragma unroll
        for (int j = 0; j < kV; ++j) v[j] = pk_add<DT>(v[j], x[j]);
        break;
      case OP_MUL_CONST: {
        const uint32_t c2 = pk_splat<DT>(c.imm[k]);
#pragma unroll
        for (int j = 0; j < kV; ++j) v[j] = pk_mul<DT>(v[j], c2);
        break;
      }
      case OP_ADD_CONST: {
        const uint32_t c2 = pk_splat<DT>(c.imm[k]);
#pragma unroll
        for (int j = 0; j < kV; ++j) v[j] = pk_add<DT>(v[j], c2);
        break;
      }
      case OP_NEG:
#pragma unroll
        for (int j = 0; j < kV; ++j) v[j] ^= 0x80008000u;
        break;
      case OP_ABS:
#pragma unroll
        for (int j = 0; j < kV; ++j) v[j] &= 0x7FFF7FFFu;
        break;
      case OP_TANH:
        if (TT && DT == BF16) {
#pragma unroll
          for (int j = 0; j < kV; ++j) v[j] = tanh_bf16x2_tab(v[j], ttab);
        } else if (OOL) {
#pragma unroll
          for (int j = 0; j < kV; ++j) v[j] = fn2_call<DT>(OP_TANH, v[j], lt);
        } else {
          fn16x2<DT, OP_TANH, kV>(v, lt);
        }
        break;
      default:  // exp, log
        if (TT && DT == BF16) {
          // not reached: chains with a table tanh have no exp or log
        } else if (OOL) {
          const int op = c.op[k];
#pragma unroll
          for (int j = 0; j < kV; ++j) v[j] = fn2_call<DT>(op, v[j], lt);
        } else if (c.op[k] == OP_EXP) {
          fn16x2<DT, OP_EXP, kV>(v, lt);
        } else {
          fn16x2<DT, OP_LOG, kV>(v, lt);
        }
    }
  }
}

// Streaming kernel: a thread takes four 16-byte vectors (32 elements) per step -- a warp 2 KiB of
// contiguous input, each of its four loads 512 contiguous bytes -- and runs the chain on them with one
// op dispatch per 32 elements; the vectors left after the last full round of steps go one per thread,
// so no thread ends more than one vector behind another. With TT (a bf16 chain with tanh) each block
// copies the 64 KiB tanh table into its shared memory while its first loads are in flight.
constexpr int kTanhTabThreads = 1024;
template <int DT, bool TT>
__global__ void __launch_bounds__(TT ? kTanhTabThreads : 256, TT ? 1 : 4) elementwise_16x2_kernel(EwPlan p) {
  const LogTab lt = global_log_tables();
  extern __shared__ __align__(16) uint16_t ttab[];
  const uint4* in = reinterpret_cast<const uint4*>(p.in);
  uint4* out = reinterpret_cast<uint4*>(p.out);
  const int64_t nvec = p.n / 8;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t lane = threadIdx.x & 31, gwarp = gtid >> 5;
  const int64_t rounds = nvec / (4 * nthreads);
  uint32_t x[16];
  auto load4 = [&](int64_t r) {
    const int64_t b = r * 4 * nthreads + gwarp * 128 + lane;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint4 w = __ldg(in + b + 32 * u);
      x[4 * u] = w.x, x[4 * u + 1] = w.y, x[4 * u + 2] = w.z, x[4 * u + 3] = w.w;
    }
  };
  if (rounds > 0) load4(0);
  if (TT) {
    for (int i = threadIdx.x; i < 32768 / 8; i += blockDim.x)
      reinterpret_cast<uint4*>(ttab)[i] = reinterpret_cast<const uint4*>(kTanhBf16)[i];
    __syncthreads();
  }
  for (int64_t r = 0; r < rounds; ++r) {
    if (r > 0) load4(r);
    uint32_t v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = x[j];
    chain16x2<DT, 16, TT, true>(p.pro, v, x, lt, ttab);
    const int64_t b = r * 4 * nthreads + gwarp * 128 + lane;
#pragma unroll
    for (int u = 0; u < 4; ++u) out[b + 32 * u] = make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
  }
  for (int64_t i = rounds * 4 * nthreads + gtid; i < nvec; i += nthreads) {
    const uint4 w = __ldg(in + i);
    const uint32_t y[4] = {w.x, w.y, w.z, w.w};
    uint32_t v[4] = {w.x, w.y, w.z, w.w};
    chain16x2<DT, 4, TT, true>(p.pro, v, y, lt, ttab);
    out[i] = make_uint4(v[0], v[1], v[2], v[3]);
  }
  for (int64_t e = nvec * 8 + gtid; e < p.n; e += nthreads) {
    const float r = apply_chain_rt(p.pro, load_as_f32(p.in, DT, e), 0, lt);
    store_from_f32(p.out, DT, e, r);
  }
}

// True when the 16-bit vector kernel applies: every op rounded to the 16-bit type, no broadcast
// operand, no epilogue.
static bool chain16x2_ok(const Chain& pro, const Chain& epi, int dt) {
  if ((dt != BF16 && dt != F16) || epi.n != 0 || !pro.round16) return false;
  for (int k = 0; k < pro.n; ++k)
    if (pro.op[k] == OP_ADD_BCAST) return false;
  return true;
}

// ---- 16-bit chains as a table of all 65536 inputs ------------------------------------------------
// A chain on a 16-bit input with a 16-bit result (no broadcast operand) is a function of the input's
// bits alone, so a large input is served from a table of its 65536 results held in shared memory
// (128 KiB per block, one block of 1024 threads per SM). The blocks of a thread-block cluster (8 where
// they fit) build the table together: each evaluates its share of the entries with the per-element
// code and writes them into the shared memory of every block of its cluster (distributed shared
// memory); after the cluster barrier each block streams 16-byte vectors and looks every element up
// locally. No global memory beyond input and output.
constexpr int kLutThreads = 1024;
constexpr int64_t kJitMinElems = int64_t(1) << 20;  // smaller chains stay with the interpreter kernels
constexpr int kLutEntries = 1 << 16;
constexpr int64_t kLutMinElems = int64_t(1) << 22;  // below this the direct kernels are faster

template <int DT>
__device__ __forceinline__ uint32_t lut_entry(const EwPlan& p, uint32_t bits, const LogTab& lt) {
  const float x = DT == BF16 ? bf16_bits_to_f32(bits) : f16_bits_to_f32((uint16_t)bits);
  const float v = round_to_dt(ew_apply(p, x, lt), DT);
  return DT == BF16 ? f32_to_bf16_bits(v) : f32_to_f16_bits(v);
}

__device__ __forceinline__ uint32_t lut_pair(const uint16_t* lut, uint32_t w) {
  return (uint32_t)lut[w & 0xFFFFu] | ((uint32_t)lut[w >> 16] << 16);
}

// PACKED: the chain qualifies for the packed pair evaluation (chain16x2), used for the table too.
template <int DT, bool PACKED>
__global__ void __launch_bounds__(kLutThreads, 1) elementwise_lut16_kernel(EwPlan p) {
  extern __shared__ __align__(16) uint16_t lut[];  // kLutEntries results
  cg::cluster_group cluster = cg::this_cluster();
  const LogTab lt = global_log_tables();
  const int nb = (int)cluster.num_blocks(), share = kLutEntries / nb;
  for (int c = 8 * (int)threadIdx.x; c < share; c += 8 * kLutThreads) {
    // this block's share of the table, eight consecutive entries at a time, copied to every block
    const int first = (int)cluster.block_rank() * share + c;
    uint32_t w[4];
    if (PACKED) {
      uint32_t x[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = w[i] = (uint32_t)(first + 2 * i) | ((uint32_t)(first + 2 * i + 1) << 16);
      chain16x2<DT, 4>(p.pro, w, x, lt);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = lut_entry<DT>(p, first + 2 * i, lt) | (lut_entry<DT>(p, first + 2 * i + 1, lt) << 16);
    }
    const uint4 v = make_uint4(w[0], w[1], w[2], w[3]);
    for (int d = 0; d < nb; ++d) *reinterpret_cast<uint4*>(cluster.map_shared_rank(lut, d) + first) = v;
  }
  cluster.sync();  // every block's table is complete; no shared-memory access crosses blocks after this
  const uint16_t* in = reinterpret_cast<const uint16_t*>(p.in);
  uint16_t* out = reinterpret_cast<uint16_t*>(p.out);
  const int64_t nv = p.n / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  constexpr int kU = 4;  // vectors in flight per thread
  for (int64_t v0 = tid; v0 < nv; v0 += kU * stride) {
    uint4 x[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < nv)
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(x[u].x), "=r"(x[u].y), "=r"(x[u].z), "=r"(x[u].w)
                     : "l"(reinterpret_cast<const uint4*>(in) + v));
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t v = v0 + u * stride;
      if (v < nv)
        reinterpret_cast<uint4*>(out)[v] =
            make_uint4(lut_pair(lut, x[u].x), lut_pair(lut, x[u].y), lut_pair(lut, x[u].z), lut_pair(lut, x[u].w));
    }
  }
  for (int64_t e = nv * 8 + tid; e < p.n; e += stride) out[e] = lut[in[e]];
}

// The table pays for a large input whose chain has an op the packed kernel evaluates slowly: exp or
// log, or tanh other than on bf16 values (the packed kernel reads bf16 tanh from kTanhBf16).
static bool lut16_ok(const Chain& pro, const Chain& epi, int dt, int64_t n) {
  if ((dt != BF16 && dt != F16) || n < kLutMinElems) return false;
  const bool tanh_tab = dt == BF16 && chain16x2_ok(pro, epi, dt);
  bool costly = false;
  for (const Chain* c : {&pro, &epi})
    for (int k = 0; k < c->n; ++k) {
      if (c->op[k] == OP_ADD_BCAST) return false;
      if (c->op[k] == OP_EXP || c->op[k] == OP_LOG || (c->op[k] == OP_TANH && !tanh_tab)) costly = true;
    }
  return costly;
}

// The packed 16-bit kernel, with the tanh table when a bf16 chain has tanh (and no exp or log):
// 1024-thread blocks, one per SM; otherwise 256-thread blocks. Either way the grid is one full wave
// of resident blocks (or fewer when the input is small).
template <int DT>
static cudaError_t launch_16x2(const EwPlan& p, cudaStream_t s) {
  bool tanh = false, explog = false;
  for (int k = 0; k < p.pro.n; ++k) {
    tanh |= p.pro.op[k] == OP_TANH;
    explog |= p.pro.op[k] == OP_EXP || p.pro.op[k] == OP_LOG;
  }
  constexpr bool kTab = DT == BF16;  // the table variant exists for bf16 only
  const bool tt = kTab && tanh && !explog;
  const int threads = tt ? kTanhTabThreads : 256;
  const size_t smem = tt ? 32768 * sizeof(uint16_t) : 0;
  const void* kernel = tt ? (const void*)elementwise_16x2_kernel<DT, kTab> : (const void*)elementwise_16x2_kernel<DT, false>;
  int64_t blocks = (p.n / 32 + threads - 1) / threads;
  const int64_t cap = (int64_t)device_sm_count() * kernel_blocks_per_sm(kernel, threads, smem);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (tt) elementwise_16x2_kernel<DT, kTab><<<(unsigned)blocks, threads, smem, s>>>(p);
  else elementwise_16x2_kernel<DT, false><<<(unsigned)blocks, threads, 0, s>>>(p);
  return cudaGetLastError();
}

template <int DT, bool PACKED>
static cudaError_t lut16_launch(const EwPlan& p, cudaStream_t s) {
  const size_t smem = kLutEntries * sizeof(uint16_t);
  auto kernel = elementwise_lut16_kernel<DT, PACKED>;
  int cs = 0, clusters = 0;
  table_cluster_shape((const void*)kernel, kLutThreads, smem, &cs, &clusters);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(cs * (clusters > 0 ? clusters : 1)), 1, 1);
  cfg.blockDim = dim3(kLutThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Pure data movement with identical memory order: raw bytes, 16 at a time where aligned.
__global__ void __launch_bounds__(256) copy_bytes_kernel(const uint8_t* in, uint8_t* out, int64_t nbytes, bool vec) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t done = 0;
  if (vec) {
    const int64_t nv = nbytes / 16;
    for (int64_t v = tid; v < nv; v += stride)
      reinterpret_cast<uint4*>(out)[v] = __ldg(reinterpret_cast<const uint4*>(in) + v);
    done = nv * 16;
  }
  for (int64_t b = done + tid; b < nbytes; b += stride) out[b] = in[b];
}

cudaError_t launch_copy(const void* in, void* out, int64_t nbytes, cudaStream_t s) {
  if (nbytes == 0) return cudaSuccess;
  int64_t blocks = (nbytes + 4095) / 4096;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const bool vec = ((uintptr_t)in % 16 == 0) && ((uintptr_t)out % 16 == 0);
  copy_bytes_kernel<<<(unsigned)blocks, 256, 0, s>>>(reinterpret_cast<const uint8_t*>(in),
                                                      reinterpret_cast<uint8_t*>(out), nbytes, vec);
  return cudaGetLastError();
}

const void* tanh_table_address() {
  static std::mutex mu;
  static std::map<int, const void*> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  void* p = nullptr;
  const cudaError_t pending = cudaPeekAtLastError();
  if (cudaGetSymbolAddress(&p, kTanhBf16) != cudaSuccess) {
    p = nullptr;
    if (pending == cudaSuccess) cudaGetLastError();  // the query's own error
  }
  cache[dev] = p;
  return p;
}

cudaError_t launch_elementwise(const void* in, void* out, int64_t n, int dt, const Chain& pro, const Chain& epi,
                               cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  // large 16-bit chains the generator covers: a kernel written for the chain (jit_chain.cu)
  if (n >= kJitMinElems && jit_chain_ok(pro, epi, dt) && (uintptr_t)in % 16 == 0 && (uintptr_t)out % 16 == 0) {
    bool used = false;
    const cudaError_t e = launch_jit_chain(in, out, n, dt, pro, s, &used);
    if (e != cudaSuccess || used) return e;
  }
  EwPlan p{in, out, n, dt, pro, epi};
  int64_t blocks = (n + 1023) / 1024;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (dt == F32) {
    const bool vec = ((uintptr_t)in % 16 == 0) && ((uintptr_t)out % 16 == 0);
    if (vec) elementwise_f32_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(p);
    else elementwise_f32_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(p);
  } else if (lut16_ok(pro, epi, dt, n) && (uintptr_t)in % 16 == 0 && (uintptr_t)out % 16 == 0) {
    if (chain16x2_ok(pro, epi, dt)) return dt == BF16 ? lut16_launch<BF16, true>(p, s) : lut16_launch<F16, true>(p, s);
    return dt == BF16 ? lut16_launch<BF16, false>(p, s) : lut16_launch<F16, false>(p, s);
  } else if (chain16x2_ok(pro, epi, dt) && (uintptr_t)in % 16 == 0 && (uintptr_t)out % 16 == 0) {
    return dt == BF16 ? launch_16x2<BF16>(p, s) : launch_16x2<F16>(p, s);
  } else {
    elementwise_any_kernel<<<(unsigned)blocks, 256, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace hlo
