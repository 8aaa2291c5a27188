// Plain CPU oracle for HLO hero fusions (reduce, transpose, layout change, uniform quantization).
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls this file; only the
// test suite, the package smoke check and the benchmark's CPU-baseline leg use it. It shares no code,
// header, table or constant with the CUDA library: every rule below is re-derived from the pages.
//
// Written to be read against the pages, not to be fast:
//   * Layout addressing follows "XLA Shapes and Layout", section "Layout" (minor_to_major: the first
//     entry is the minor-most dimension, the one that changes fastest in linear memory) and
//     "Default minor-to-major ordering" ([N-1, ..., 0]).
//   * reduce follows "StableHLO Specification", section "reduce": every output element is the
//     reduction of its slice, the slice visited in ascending lexicographic index order (the in-order
//     traversal the spec requires of any schedule), with the init value applied once, as in the
//     pseudocode of "XLA Operation Semantics", section "Reduce".
//   * Elementwise ops (exponential, log, abs, negate, add) follow the spec's op sections: IEEE-754
//     operations whose result type equals the operand type (constraint C1 of each op), so every op
//     result is the correctly rounded value in the element type.
//   * broadcast_in_dim follows its spec section: operand_index[d] = 0 if dim(operand, d) = 1, else
//     result_index[broadcast_dimensions[d]].
//   * maximum is IEEE-754 maximum (NaN propagates, -0 < +0), spec section "maximum".
//   * Transpose: result[r] = operand[i] with i[permutation[k]] = r[k], the output-to-input indexing
//     map of "XLA:GPU Emitters", section "Indexing transformations" ([20,40] -> [40,20] reads
//     (d0, d1) -> (d1, d0)).
//   * Quantization: real = scale * (q - zero_point) ("StableHLO Quantization", uniform quantization;
//     spec section "Types", quantized element types), per-tensor or per-axis along
//     quantization_dimension; quantize = clamp(round_nearest_even(real / scale) + zero_point,
//     storage_min, storage_max) in the expressed type f32.
//
// Floating point: reductions accumulate in f64; elementwise ops are evaluated in f64 (or long double
// where the f64 value lies within 2^-50 relative of a rounding boundary of the element type) and
// rounded once to the element type; the quantization chain is evaluated in f32 IEEE operations because its expressed
// type is f32. Build with -O2 -fno-fast-math -ffp-contract=off so that no operation is contracted.
//
// Parallelism: OpenMP over independent output elements only; no cross-thread reduction, so results do
// not depend on the thread count.

#include <cfenv>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <limits>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

// Exported functions carry extern "C"; everything else has internal linkage.

// ----------------------------------------------------------------------------------------------
// Descriptors (the oracle's own; plain C layout, mirrored by oracle/__init__.py with ctypes).
// ----------------------------------------------------------------------------------------------
enum { ORC_MAX_RANK = 8, ORC_MAX_OPS = 16 };
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_S8 = 2, ORC_F16 = 3, ORC_S32 = 4, ORC_F64 = 5, ORC_U8 = 6 };
enum {
  ORC_OP_EXP = 1, ORC_OP_LOG = 2, ORC_OP_ABS = 3, ORC_OP_NEG = 4, ORC_OP_ADD_BCAST = 5, ORC_OP_TANH = 6,
  ORC_OP_ADD_CONST = 7, ORC_OP_MUL_CONST = 8, ORC_OP_ADD_INPUT = 9, ORC_OP_MUL_INPUT = 10
};
enum { ORC_RED_ADD = 0, ORC_RED_MAX = 1 };
enum { ORC_OK = 0, ORC_EINVAL = 1, ORC_EUNRESOLVED = 2 };

typedef struct {
  int32_t rank;
  int32_t dtype;
  int64_t dims[ORC_MAX_RANK];
  int64_t m2m[ORC_MAX_RANK];  // minor_to_major
} orc_arr;

typedef struct {
  int32_t n_ops;
  int32_t ops[ORC_MAX_OPS];
  // 1: every op result is rounded to the element type of the operand (the spec's types);
  // 0: for 16-bit float operands, intermediates are kept in f32 instead.
  int32_t round_each;
  int32_t has_bcast;
  orc_arr bcast;                            // the broadcast operand of ORC_OP_ADD_BCAST
  int64_t bcast_dimensions[ORC_MAX_RANK];   // broadcast_in_dim's broadcast_dimensions
  const void* bcast_data;
  // ORC_OP_ADD_CONST / ORC_OP_MUL_CONST: the constant, taken as a value of the element type
  // ("StableHLO Specification", "constant"); ORC_OP_ADD_INPUT / MUL_INPUT combine the running value
  // with the element that entered the chain.
  double imm[ORC_MAX_OPS];
} orc_chain;

typedef struct {
  int32_t per_axis;            // 0: per-tensor (one scale/zero point), 1: per-axis
  int32_t quantization_dimension;
  int64_t n;                   // number of (scale, zero_point) pairs
  const float* scales;
  const int32_t* zero_points;
  int32_t storage_min;
  int32_t storage_max;
} orc_quant;

// Number of elements each dtype code occupies, in bytes.
static int elem_bytes(int dt) {
  switch (dt) {
    case ORC_F32: return 4;
    case ORC_BF16: return 2;
    case ORC_S8: return 1;
    case ORC_U8: return 1;
    case ORC_F16: return 2;
    case ORC_S32: return 4;
    case ORC_F64: return 8;
  }
  return 0;
}

// ----------------------------------------------------------------------------------------------
// Layout addressing ("XLA Shapes and Layout", section "Layout").
// The minor-most dimension m2m[0] has stride 1; each next dimension in minor_to_major order has the
// stride of the previous one times the previous one's size.
// ----------------------------------------------------------------------------------------------
static void strides_of(const orc_arr* a, int64_t* stride) {
  int64_t s = 1;
  for (int k = 0; k < a->rank; ++k) {
    stride[a->m2m[k]] = s;
    s *= a->dims[a->m2m[k]];
  }
}

static int64_t num_elements(const orc_arr* a) {
  int64_t n = 1;
  for (int d = 0; d < a->rank; ++d) n *= a->dims[d];
  return n;
}

static bool valid_arr(const orc_arr* a) {
  if (!a || a->rank < 0 || a->rank > ORC_MAX_RANK || elem_bytes(a->dtype) == 0) return false;
  bool seen[ORC_MAX_RANK] = {false};
  for (int k = 0; k < a->rank; ++k) {
    int64_t d = a->m2m[k];
    if (d < 0 || d >= a->rank || seen[d]) return false;
    seen[d] = true;
    if (a->dims[k] < 0) return false;
  }
  return true;
}

// Linear offset (in elements) of logical index idx in array a.
extern "C" int orc_linear_offset(const orc_arr* a, const int64_t* idx, int64_t* out) {
  if (!valid_arr(a)) return ORC_EINVAL;
  int64_t stride[ORC_MAX_RANK];
  strides_of(a, stride);
  int64_t off = 0;
  for (int d = 0; d < a->rank; ++d) {
    if (idx[d] < 0 || idx[d] >= a->dims[d]) return ORC_EINVAL;
    off += idx[d] * stride[d];
  }
  *out = off;
  return ORC_OK;
}

// Logical index of the n-th element in ascending lexicographic order (last dimension fastest).
static void lex_index(int rank, const int64_t* dims, int64_t n, int64_t* idx) {
  for (int d = rank - 1; d >= 0; --d) {
    int64_t sz = dims[d];
    idx[d] = sz > 0 ? n % sz : 0;
    n = sz > 0 ? n / sz : 0;
  }
}

// ----------------------------------------------------------------------------------------------
// Rounding to a binary floating-point format with round-to-nearest, ties to even.
// prec = significand bits (24 for f32, 8 for bf16, 11 for f16), emin/emax = exponent range.
// ----------------------------------------------------------------------------------------------
template <typename T>
static T round_to_format(T v, int prec, int emin, int emax) {
  if (v == 0 || std::isnan(v) || std::isinf(v)) return v;
  int e;
  std::frexp(v, &e);            // v = f * 2^e, 0.5 <= |f| < 1, so the leading bit has weight 2^(e-1)
  int lead = e - 1;
  if (lead < emin) lead = emin;  // gradual underflow: fixed quantum below the normal range
  T quantum = std::ldexp((T)1, lead - prec + 1);
  T scaled = v / quantum;          // exact: division by a power of two
  T r = std::nearbyint(scaled);    // default rounding mode: ties to even
  T out = r * quantum;
  T maxv = std::ldexp((T)1, emax) * (2 - std::ldexp((T)1, 1 - prec));
  if (std::fabs(out) > maxv) return v > 0 ? INFINITY : -INFINITY;
  return out;
}

// Distance-to-boundary test: true when v lies within rel*|v| of a rounding boundary (a midpoint
// between two neighbours) of the format, so that an approximation of v with that relative error
// could round either way.
template <typename T>
static bool near_boundary(T v, int prec, int emin, T rel) {
  if (v == 0 || std::isnan(v) || std::isinf(v)) return false;
  int e;
  std::frexp(v, &e);
  int lead = e - 1;
  if (lead < emin) lead = emin;
  T quantum = std::ldexp((T)1, lead - prec + 1);
  T scaled = v / quantum;                 // exact
  T frac = scaled - std::floor(scaled);   // position between two representable neighbours (exact)
  T tol = std::fabs(v) * rel / quantum;
  return std::fabs(frac - (T)0.5) <= tol;
}

static int prec_of(int dt) { return dt == ORC_BF16 ? 8 : dt == ORC_F16 ? 11 : dt == ORC_F64 ? 53 : 24; }
static int emin_of(int dt) { return dt == ORC_F16 ? -14 : dt == ORC_F64 ? -1022 : -126; }
static int emax_of(int dt) { return dt == ORC_F16 ? 15 : dt == ORC_F64 ? 1023 : 127; }

static bool is_float_type(int dt) { return dt == ORC_F32 || dt == ORC_BF16 || dt == ORC_F16 || dt == ORC_F64; }

// Rounds v into element type dt. Integer types hold their values exactly (a transpose or layout change
// moves elements; it does not convert them), so nothing is rounded for them.
template <typename T>
static T round_to(T v, int dt) {
  if (!is_float_type(dt)) return v;
  if (dt == ORC_F64) return (T)(double)v;
  return round_to_format<T>(v, prec_of(dt), emin_of(dt), emax_of(dt));
}

// Elements that could not be rounded with certainty even in long double are counted here.
static int g_unresolved = 0;

// Correctly rounded exp / log into format dt. The f64 libm value (error well under one f64 ulp) is
// trusted unless it lies close to a rounding boundary of dt; then long double decides.
static double cr_exp(double x, int dt) {
  double d = std::exp(x);
  if (!near_boundary<double>(d, prec_of(dt), emin_of(dt), std::ldexp(1.0, -50))) return round_to<double>(d, dt);
  long double l = std::exp((long double)x);
  if (near_boundary<long double>(l, prec_of(dt), emin_of(dt), std::ldexp(1.0L, -60))) {
#pragma omp atomic
    g_unresolved++;
  }
  return (double)round_to<long double>(l, dt);
}

static double cr_log(double x, int dt) {
  if (std::isnan(x)) return x;
  if (x < 0) return NAN;                 // IEEE log of a negative number: invalid
  if (x == 0) return -INFINITY;          // log(+-0) = -inf
  if (std::isinf(x)) return INFINITY;
  double d = std::log(x);
  if (!near_boundary<double>(d, prec_of(dt), emin_of(dt), std::ldexp(1.0, -50))) return round_to<double>(d, dt);
  long double l = std::log((long double)x);
  if (near_boundary<long double>(l, prec_of(dt), emin_of(dt), std::ldexp(1.0L, -60))) {
#pragma omp atomic
    g_unresolved++;
  }
  return (double)round_to<long double>(l, dt);
}

// Correctly rounded tanh ("StableHLO Specification", "tanh": IEEE-754 tanh of the element type), the
// same way: libm's double tanh, rechecked in long double next to a rounding boundary.
static double cr_tanh(double x, int dt) {
  if (std::isnan(x)) return x;
  double d = std::tanh(x);
  if (!near_boundary<double>(d, prec_of(dt), emin_of(dt), std::ldexp(1.0, -50))) return round_to<double>(d, dt);
  long double l = std::tanh((long double)x);
  if (near_boundary<long double>(l, prec_of(dt), emin_of(dt), std::ldexp(1.0L, -60))) {
#pragma omp atomic
    g_unresolved++;
  }
  return (double)round_to<long double>(l, dt);
}

extern "C" int orc_unresolved_count(void) { return g_unresolved; }
extern "C" void orc_reset_unresolved(void) { g_unresolved = 0; }

// ----------------------------------------------------------------------------------------------
// Element loads and stores.
// ----------------------------------------------------------------------------------------------
static double load_elem(const void* base, int dt, int64_t off) {
  switch (dt) {
    case ORC_F32: { float v; std::memcpy(&v, (const char*)base + off * 4, 4); return v; }
    case ORC_F64: { double v; std::memcpy(&v, (const char*)base + off * 8, 8); return v; }
    case ORC_BF16: {  // bf16 holds the upper 16 bits of an f32
      uint16_t h; std::memcpy(&h, (const char*)base + off * 2, 2);
      uint32_t u = (uint32_t)h << 16; float v; std::memcpy(&v, &u, 4); return v;
    }
    case ORC_F16: {
      uint16_t h; std::memcpy(&h, (const char*)base + off * 2, 2);
      int sign = h >> 15, ex = (h >> 10) & 31, man = h & 1023;
      double v;
      if (ex == 0) v = std::ldexp((double)man, -24);
      else if (ex == 31) v = man ? NAN : INFINITY;
      else v = std::ldexp((double)(man + 1024), ex - 25);
      return sign ? -v : v;
    }
    case ORC_S8: return (double)((const int8_t*)base)[off];
    case ORC_U8: return (double)((const uint8_t*)base)[off];
    case ORC_S32: return (double)((const int32_t*)base)[off];
  }
  return 0;
}

// Stores v, which must already be representable in dt (callers round first).
static void store_elem(void* base, int dt, int64_t off, double v) {
  switch (dt) {
    case ORC_F32: { float f = (float)v; std::memcpy((char*)base + off * 4, &f, 4); return; }
    case ORC_F64: { double f = (double)v; std::memcpy((char*)base + off * 8, &f, 8); return; }
    case ORC_BF16: {
      float f = (float)v; uint32_t u; std::memcpy(&u, &f, 4);
      uint16_t h = (uint16_t)(u >> 16);
      if (std::isnan(v)) h = 0x7FC0;  // canonical quiet NaN
      std::memcpy((char*)base + off * 2, &h, 2); return;
    }
    case ORC_F16: {
      uint16_t h;
      if (std::isnan(v)) h = 0x7E00;
      else {
        int sign = std::signbit(v) ? 1 : 0;
        double a = std::fabs(v);
        if (std::isinf(a)) h = 0x7C00;
        else if (a < std::ldexp(1.0, -14)) h = (uint16_t)(long)(a * std::ldexp(1.0, 24));
        else { int e; double m = std::frexp(a, &e); h = (uint16_t)(((e + 14) << 10) | ((long)(m * 2048) - 1024)); }
        h |= (uint16_t)(sign << 15);
      }
      std::memcpy((char*)base + off * 2, &h, 2); return;
    }
    case ORC_S8: ((int8_t*)base)[off] = (int8_t)(long)v; return;
    case ORC_U8: ((uint8_t*)base)[off] = (uint8_t)(long)v; return;
    case ORC_S32: ((int32_t*)base)[off] = (int32_t)(long)v; return;
  }
}

// ----------------------------------------------------------------------------------------------
// broadcast_in_dim ("StableHLO Specification", section "broadcast_in_dim").
// ----------------------------------------------------------------------------------------------
static int64_t bcast_offset(const orc_chain* c, const int64_t* result_index) {
  int64_t stride[ORC_MAX_RANK];
  strides_of(&c->bcast, stride);
  int64_t off = 0;
  for (int d = 0; d < c->bcast.rank; ++d) {
    int64_t oi = c->bcast.dims[d] == 1 ? 0 : result_index[c->bcast_dimensions[d]];
    off += oi * stride[d];
  }
  return off;
}

// Materialises broadcast_in_dim(operand) into result (both described by layouts), for pinning.
extern "C" int orc_broadcast_in_dim(const orc_arr* operand, const void* operand_data,
                         const int64_t* broadcast_dimensions, const orc_arr* result, void* result_data) {
  if (!valid_arr(operand) || !valid_arr(result) || operand->dtype != result->dtype) return ORC_EINVAL;
  for (int d = 0; d < operand->rank; ++d) {
    int64_t bd = broadcast_dimensions[d];
    if (bd < 0 || bd >= result->rank) return ORC_EINVAL;
    if (operand->dims[d] != 1 && operand->dims[d] != result->dims[bd]) return ORC_EINVAL;
  }
  orc_chain c;
  std::memset(&c, 0, sizeof c);
  c.bcast = *operand;
  for (int d = 0; d < operand->rank; ++d) c.bcast_dimensions[d] = broadcast_dimensions[d];
  int64_t rstride[ORC_MAX_RANK];
  strides_of(result, rstride);
  int64_t n = num_elements(result);
  for (int64_t i = 0; i < n; ++i) {
    int64_t idx[ORC_MAX_RANK];
    lex_index(result->rank, result->dims, i, idx);
    int64_t roff = 0;
    for (int d = 0; d < result->rank; ++d) roff += idx[d] * rstride[d];
    std::memcpy((char*)result_data + roff * elem_bytes(result->dtype),
                (const char*)operand_data + bcast_offset(&c, idx) * elem_bytes(operand->dtype),
                elem_bytes(result->dtype));
  }
  return ORC_OK;
}

// ----------------------------------------------------------------------------------------------
// Elementwise chain. v is an exact value of element type dt; index is the element's logical index
// in the fused array (used by the broadcast operand). Returns a value exactly representable in the
// working type (dt under round_each, else f32 for 16-bit floats).
// ----------------------------------------------------------------------------------------------
static int working_type(const orc_chain* c, int dt) {
  if (!c || c->round_each) return dt;
  return (dt == ORC_BF16 || dt == ORC_F16) ? ORC_F32 : dt;
}

static double apply_chain(const orc_chain* c, double v, int dt, const int64_t* index) {
  if (!c) return v;
  int wt = working_type(c, dt);
  const double x = v;  // the element entering the chain
  for (int k = 0; k < c->n_ops; ++k) {
    // products and sums of two values of at most 24 significand bits: exact in double for the
    // product; a sum rounded in double first is still rounded correctly into f32/bf16/f16
    // (53 >= 2 * 24 + 2)
    const double cst = round_to<double>(c->imm[k], dt);
    switch (c->ops[k]) {
      case ORC_OP_EXP: v = cr_exp(v, wt); break;
      case ORC_OP_LOG: v = cr_log(v, wt); break;
      case ORC_OP_TANH: v = cr_tanh(v, wt); break;
      case ORC_OP_ADD_CONST: v = round_to<double>(v + cst, wt); break;
      case ORC_OP_MUL_CONST: v = round_to<double>(v * cst, wt); break;
      case ORC_OP_ADD_INPUT: v = round_to<double>(v + x, wt); break;
      case ORC_OP_MUL_INPUT: v = round_to<double>(v * x, wt); break;
      case ORC_OP_ABS: v = std::fabs(v); break;
      case ORC_OP_NEG: v = -v; break;
      case ORC_OP_ADD_BCAST: {
        double b = load_elem(c->bcast_data, c->bcast.dtype, bcast_offset(c, index));
        v = round_to<double>(v + b, wt);  // f64 sum of two short floats, then the element type: the
                                          // double rounding is innocuous (53 >= 2 * 24 + 2)
        break;
      }
      default: break;
    }
  }
  return v;
}

static bool valid_chain(const orc_chain* c, const orc_arr* fused) {
  if (!c) return true;
  if (c->n_ops < 0 || c->n_ops > ORC_MAX_OPS) return false;
  for (int k = 0; k < c->n_ops; ++k) {
    int op = c->ops[k];
    if (op < ORC_OP_EXP || op > ORC_OP_MUL_INPUT) return false;
    if (op == ORC_OP_ADD_BCAST) {
      if (!c->has_bcast || !valid_arr(&c->bcast) || !c->bcast_data) return false;
      for (int d = 0; d < c->bcast.rank; ++d) {
        int64_t bd = c->bcast_dimensions[d];
        if (bd < 0 || bd >= fused->rank) return false;
        if (c->bcast.dims[d] != 1 && c->bcast.dims[d] != fused->dims[bd]) return false;
      }
    }
  }
  return true;
}

// ----------------------------------------------------------------------------------------------
// reduce ("StableHLO Specification", section "reduce"; "XLA Operation Semantics", section "Reduce").
// out[j] = init (+) term(slice_j[0]) (+) term(slice_j[1]) (+) ... in lexicographic slice order,
// accumulated in f64 for add and with IEEE maximum for max. abs_sum (optional) receives sum |term| per output element, used by the tolerance.
// ----------------------------------------------------------------------------------------------
static double ieee_maximum(double a, double b) {
  if (std::isnan(a) || std::isnan(b)) return NAN;
  if (a == 0 && b == 0) return std::signbit(a) ? b : a;  // maximum(-0, +0) = +0
  return a > b ? a : b;
}

extern "C" int orc_reduce(const orc_arr* in, const void* in_data, const orc_chain* chain,
               const int64_t* dimensions, int n_dimensions, int kind, double init,
               const orc_arr* out, void* out_data, double* abs_sum) {
  if (!valid_arr(in) || !valid_arr(out) || !valid_chain(chain, in)) return ORC_EINVAL;
  if (kind != ORC_RED_ADD && kind != ORC_RED_MAX) return ORC_EINVAL;
  if (n_dimensions < 0 || n_dimensions > in->rank) return ORC_EINVAL;
  bool reduced[ORC_MAX_RANK] = {false};
  for (int i = 0; i < n_dimensions; ++i) {
    int64_t d = dimensions[i];
    if (d < 0 || d >= in->rank || reduced[d]) return ORC_EINVAL;  // spec C4, C5
    reduced[d] = true;
  }
  // Result shape = input shape without the reduced dimensions, in the same relative order (C7).
  int kept[ORC_MAX_RANK], nk = 0, red[ORC_MAX_RANK], nr = 0;
  for (int d = 0; d < in->rank; ++d) (reduced[d] ? red[nr++] : kept[nk++]) = d;
  if (out->rank != nk) return ORC_EINVAL;
  for (int k = 0; k < nk; ++k) if (out->dims[k] != in->dims[kept[k]]) return ORC_EINVAL;

  int64_t kdims[ORC_MAX_RANK], rdims[ORC_MAX_RANK];
  for (int k = 0; k < nk; ++k) kdims[k] = in->dims[kept[k]];
  for (int k = 0; k < nr; ++k) rdims[k] = in->dims[red[k]];
  int64_t n_out = 1, n_red = 1;
  for (int k = 0; k < nk; ++k) n_out *= kdims[k];
  for (int k = 0; k < nr; ++k) n_red *= rdims[k];

  int64_t istride[ORC_MAX_RANK], ostride[ORC_MAX_RANK];
  strides_of(in, istride);
  strides_of(out, ostride);

#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t o = 0; o < n_out; ++o) {
    int64_t kidx[ORC_MAX_RANK], ridx[ORC_MAX_RANK], full[ORC_MAX_RANK];
    lex_index(nk, kdims, o, kidx);
    for (int k = 0; k < nk; ++k) full[kept[k]] = kidx[k];
    // init_values has the inputs' element type ("reduce" C2): the init literal is a value of it
    double acc = round_to<double>(init, in->dtype), asum = 0;
    for (int64_t t = 0; t < n_red; ++t) {
      lex_index(nr, rdims, t, ridx);
      for (int k = 0; k < nr; ++k) full[red[k]] = ridx[k];
      int64_t off = 0;
      for (int d = 0; d < in->rank; ++d) off += full[d] * istride[d];
      double v = apply_chain(chain, load_elem(in_data, in->dtype, off), in->dtype, full);
      if (kind == ORC_RED_ADD) acc += v;
      else acc = ieee_maximum(acc, v);
      asum += std::fabs(v);
    }
    int64_t ooff = 0;
    for (int k = 0; k < nk; ++k) ooff += kidx[k] * ostride[k];
    store_elem(out_data, out->dtype, ooff, round_to<double>(acc, out->dtype));
    if (abs_sum) abs_sum[ooff] = (double)asum;
  }
  return ORC_OK;
}

// ----------------------------------------------------------------------------------------------
// Variadic reduce with the max/argmax body (XLA Operation Semantics, "Variadic Reduce"): inputs V
// (float) and K (s32, or the position along the single reduced dimension when k_data is NULL), init
// (I_V, I_K). For every output, the reduced indices are visited in lexicographic order and
//   f(max, argmax, value, index) = (value, index) if value >= max else (max, argmax)
// is applied from f(I_V, I_K, V_0, K_0) on, exactly as the recursion f_0, f_1, ..., f_(N-1) of the
// pages. The value is stored in V's element type (a member of V or I_V: exact), the index as s32.
// ----------------------------------------------------------------------------------------------
extern "C" int orc_reduce_max_argmax(const orc_arr* in, const void* in_data, const orc_arr* kin, const void* k_data,
                                     const int64_t* dimensions, int n_dimensions, double init_value,
                                     int64_t init_index, const orc_arr* out, void* out_data,
                                     const orc_arr* out_idx, void* out_idx_data) {
  if (!valid_arr(in) || !valid_arr(out) || !valid_arr(out_idx)) return ORC_EINVAL;
  if (!is_float_type(in->dtype) || out->dtype != in->dtype || out_idx->dtype != ORC_S32) return ORC_EINVAL;
  if (n_dimensions < 0 || n_dimensions > in->rank) return ORC_EINVAL;
  if (k_data) {
    if (!valid_arr(kin) || kin->dtype != ORC_S32 || kin->rank != in->rank) return ORC_EINVAL;
    for (int d = 0; d < in->rank; ++d) if (kin->dims[d] != in->dims[d]) return ORC_EINVAL;
  } else if (n_dimensions != 1) {
    return ORC_EINVAL;  // the implicit index runs along one dimension
  }
  bool reduced[ORC_MAX_RANK] = {false};
  for (int i = 0; i < n_dimensions; ++i) {
    int64_t d = dimensions[i];
    if (d < 0 || d >= in->rank || reduced[d]) return ORC_EINVAL;
    reduced[d] = true;
  }
  int kept[ORC_MAX_RANK], nk = 0, red[ORC_MAX_RANK], nr = 0;
  for (int d = 0; d < in->rank; ++d) (reduced[d] ? red[nr++] : kept[nk++]) = d;
  if (out->rank != nk || out_idx->rank != nk) return ORC_EINVAL;
  for (int k = 0; k < nk; ++k)
    if (out->dims[k] != in->dims[kept[k]] || out_idx->dims[k] != in->dims[kept[k]]) return ORC_EINVAL;
  int64_t kdims[ORC_MAX_RANK], rdims[ORC_MAX_RANK];
  for (int k = 0; k < nk; ++k) kdims[k] = in->dims[kept[k]];
  for (int k = 0; k < nr; ++k) rdims[k] = in->dims[red[k]];
  int64_t n_out = 1, n_red = 1;
  for (int k = 0; k < nk; ++k) n_out *= kdims[k];
  for (int k = 0; k < nr; ++k) n_red *= rdims[k];
  int64_t istride[ORC_MAX_RANK], kstride[ORC_MAX_RANK], ostride[ORC_MAX_RANK], oistride[ORC_MAX_RANK];
  strides_of(in, istride);
  if (k_data) strides_of(kin, kstride);
  strides_of(out, ostride);
  strides_of(out_idx, oistride);
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t o = 0; o < n_out; ++o) {
    int64_t kidx[ORC_MAX_RANK], ridx[ORC_MAX_RANK], full[ORC_MAX_RANK];
    lex_index(nk, kdims, o, kidx);
    for (int k = 0; k < nk; ++k) full[kept[k]] = kidx[k];
    double mx = round_to<double>(init_value, in->dtype);
    int64_t am = init_index;
    for (int64_t t = 0; t < n_red; ++t) {
      lex_index(nr, rdims, t, ridx);
      for (int k = 0; k < nr; ++k) full[red[k]] = ridx[k];
      int64_t off = 0, koff = 0;
      for (int d = 0; d < in->rank; ++d) {
        off += full[d] * istride[d];
        if (k_data) koff += full[d] * kstride[d];
      }
      const double value = load_elem(in_data, in->dtype, off);
      const int64_t index = k_data ? (int64_t)((const int32_t*)k_data)[koff] : ridx[0];
      if (value >= mx) {  // f: (value, index) if value >= max else (max, argmax)
        mx = value;
        am = index;
      }
    }
    int64_t ooff = 0, oioff = 0;
    for (int k = 0; k < nk; ++k) {
      ooff += kidx[k] * ostride[k];
      oioff += kidx[k] * oistride[k];
    }
    store_elem(out_data, out->dtype, ooff, mx);
    ((int32_t*)out_idx_data)[oioff] = (int32_t)am;
  }
  return ORC_OK;
}

// ----------------------------------------------------------------------------------------------
// Transpose fusion: out = epilogue(T(prologue(in))) or, with self_add,
// out = epilogue(prologue(in) + T(prologue(in))) where T permutes dimensions:
// dims(out)[k] = dims(in)[perm[k]] and T(x)[r] = x[i] with i[perm[k]] = r[k].
// ----------------------------------------------------------------------------------------------
extern "C" int orc_transpose(const orc_arr* in, const void* in_data, const orc_chain* prologue,
                  const int64_t* perm, int self_add, const orc_chain* epilogue,
                  const orc_arr* out, void* out_data) {
  if (!valid_arr(in) || !valid_arr(out) || in->rank != out->rank) return ORC_EINVAL;
  if (!valid_chain(prologue, in) || !valid_chain(epilogue, out)) return ORC_EINVAL;
  if (in->dtype != out->dtype) return ORC_EINVAL;
  bool seen[ORC_MAX_RANK] = {false};
  for (int k = 0; k < in->rank; ++k) {
    if (perm[k] < 0 || perm[k] >= in->rank || seen[perm[k]]) return ORC_EINVAL;
    seen[perm[k]] = true;
    if (out->dims[k] != in->dims[perm[k]]) return ORC_EINVAL;
    if (self_add && out->dims[k] != in->dims[k]) return ORC_EINVAL;
  }
  int rank = in->rank, dt = in->dtype;
  int64_t istride[ORC_MAX_RANK], ostride[ORC_MAX_RANK];
  strides_of(in, istride);
  strides_of(out, ostride);
  int64_t n = num_elements(out);
  int wt = working_type(prologue, dt);
#pragma omp parallel for schedule(static)
  for (int64_t o = 0; o < n; ++o) {
    int64_t r[ORC_MAX_RANK], i[ORC_MAX_RANK];
    lex_index(rank, out->dims, o, r);
    for (int k = 0; k < rank; ++k) i[perm[k]] = r[k];
    int64_t ioff = 0, roff_in = 0, ooff = 0;
    for (int d = 0; d < rank; ++d) {
      ioff += i[d] * istride[d];
      roff_in += r[d] * istride[d];
      ooff += r[d] * ostride[d];
    }
    double t = apply_chain(prologue, load_elem(in_data, dt, ioff), dt, i);
    double v = t;
    if (self_add) {
      double s = apply_chain(prologue, load_elem(in_data, dt, roff_in), dt, r);
      v = round_to<double>(s + t, wt);  // add of two values of the working type, rounded once
    }
    v = apply_chain(epilogue, v, dt, r);
    store_elem(out_data, out->dtype, ooff, round_to<double>(v, dt));
  }
  return ORC_OK;
}

// ----------------------------------------------------------------------------------------------
// Layout conversion: same logical array, new minor_to_major. out[off_out(i)] = in[off_in(i)].
// ----------------------------------------------------------------------------------------------
extern "C" int orc_layout_convert(const orc_arr* in, const void* in_data, const int64_t* out_m2m, void* out_data) {
  if (!valid_arr(in)) return ORC_EINVAL;
  orc_arr out = *in;
  for (int k = 0; k < in->rank; ++k) out.m2m[k] = out_m2m[k];
  if (!valid_arr(&out)) return ORC_EINVAL;
  int64_t istride[ORC_MAX_RANK], ostride[ORC_MAX_RANK];
  strides_of(in, istride);
  strides_of(&out, ostride);
  int eb = elem_bytes(in->dtype);
  int64_t n = num_elements(in);
#pragma omp parallel for schedule(static)
  for (int64_t e = 0; e < n; ++e) {
    int64_t idx[ORC_MAX_RANK];
    lex_index(in->rank, in->dims, e, idx);
    int64_t io = 0, oo = 0;
    for (int d = 0; d < in->rank; ++d) { io += idx[d] * istride[d]; oo += idx[d] * ostride[d]; }
    std::memcpy((char*)out_data + oo * eb, (const char*)in_data + io * eb, eb);
  }
  return ORC_OK;
}

// ----------------------------------------------------------------------------------------------
// Uniform quantization.
// dequantize: real = scale[j] * (q - zero_point[j]) in f32, j = index along quantization_dimension
// (or 0 per-tensor); the integer difference is exact and the f32 product is rounded once.
// quantize: clamp(round_nearest_even(real / scale[j]) + zero_point[j], storage_min, storage_max),
// f32 IEEE division, rounding to an integral value with ties to even, then the zero point, then the
// clamp. NaN reals (not produced by the fused chains here) are mapped to the zero point.
// ----------------------------------------------------------------------------------------------
static bool valid_quant(const orc_quant* q, const orc_arr* a) {
  if (!q) return false;
  if (q->per_axis) {
    if (q->quantization_dimension < 0 || q->quantization_dimension >= a->rank) return false;
    if (q->n != a->dims[q->quantization_dimension]) return false;  // C13
  } else if (q->n != 1) {
    return false;                                                  // C11
  }
  if (q->storage_min >= q->storage_max) return false;              // C4
  for (int64_t i = 0; i < q->n; ++i) {
    float s = q->scales[i];
    if (!(s > 0) || !std::isfinite(s)) return false;               // C6, C7
    if (q->zero_points[i] < q->storage_min || q->zero_points[i] > q->storage_max) return false;  // C8
  }
  return true;
}

static float dequantize_one(const orc_quant* q, int32_t code, const int64_t* idx) {
  int64_t j = q->per_axis ? idx[q->quantization_dimension] : 0;
  int32_t diff = code - q->zero_points[j];  // exact integer subtraction
  float real = q->scales[j] * (float)diff;  // one f32 multiply
  return real;
}

static int32_t quantize_one(const orc_quant* q, float real, const int64_t* idx) {
  int64_t j = q->per_axis ? idx[q->quantization_dimension] : 0;
  if (std::isnan(real)) return q->zero_points[j];
  float ratio = real / q->scales[j];        // IEEE f32 division
  float rounded = std::nearbyint(ratio);    // round to integral, ties to even (default mode)
  float shifted = rounded + (float)q->zero_points[j];
  if (shifted < (float)q->storage_min) shifted = (float)q->storage_min;
  if (shifted > (float)q->storage_max) shifted = (float)q->storage_max;
  return (int32_t)shifted;
}

// dequant(in) -> float chain (f32) -> relayout to out->m2m -> quant(out_q), or f32 out if out_q is
// NULL. out->dims must equal in->dims (a layout change keeps the logical shape).
extern "C" int orc_quant_fusion(const orc_arr* in, const void* in_data, const orc_quant* in_q,
                     const orc_chain* float_ops, const orc_arr* out, void* out_data,
                     const orc_quant* out_q) {
  if (!valid_arr(in) || !valid_arr(out) || in->rank != out->rank) return ORC_EINVAL;
  if (!valid_quant(in_q, in)) return ORC_EINVAL;
  if (out_q && !valid_quant(out_q, out)) return ORC_EINVAL;
  if (!out_q && out->dtype != ORC_F32) return ORC_EINVAL;
  if (!valid_chain(float_ops, in)) return ORC_EINVAL;
  for (int d = 0; d < in->rank; ++d) if (in->dims[d] != out->dims[d]) return ORC_EINVAL;
  int64_t istride[ORC_MAX_RANK], ostride[ORC_MAX_RANK];
  strides_of(in, istride);
  strides_of(out, ostride);
  int64_t n = num_elements(in);
#pragma omp parallel for schedule(static)
  for (int64_t e = 0; e < n; ++e) {
    int64_t idx[ORC_MAX_RANK];
    lex_index(in->rank, in->dims, e, idx);
    int64_t io = 0, oo = 0;
    for (int d = 0; d < in->rank; ++d) { io += idx[d] * istride[d]; oo += idx[d] * ostride[d]; }
    int32_t code = (int32_t)load_elem(in_data, in->dtype, io);
    float real = dequantize_one(in_q, code, idx);
    real = (float)apply_chain(float_ops, real, ORC_F32, idx);
    if (out_q) store_elem(out_data, out->dtype, oo, (double)quantize_one(out_q, real, idx));
    else store_elem(out_data, ORC_F32, oo, real);
  }
  return ORC_OK;
}

// ----------------------------------------------------------------------------------------------
// Data movement of quantized tensors: broadcast_in_dim and reshape ("StableHLO Specification",
// sections "broadcast_in_dim" and "reshape"). Both copy stored values (result[result_index] =
// operand[operand_index]); the quantization parameters of the result follow from the constraints:
//   broadcast_in_dim (C1, C6): a per-tensor operand gives a per-tensor result with the same
//     (scale, zero_point); a per-axis operand along qd gives a per-axis result along
//     broadcast_dimensions[qd], whose parameters are the operand's, or, when dim(operand, qd) = 1,
//     the operand's single pair repeated dim(result, broadcast_dimensions[qd]) times;
//   reshape (C1, C3): the parameters are unchanged; for a per-axis operand the result's quantization
//     dimension must keep the quantized axis intact -- the same size, the same product of the
//     dimensions before it and the same product of the dimensions after it.
// ----------------------------------------------------------------------------------------------
extern "C" int orc_quant_broadcast_in_dim(const orc_arr* operand, const void* operand_data, const orc_quant* q,
                                          const int64_t* broadcast_dimensions, const orc_arr* result,
                                          void* result_data, float* result_scales, int32_t* result_zero_points,
                                          int32_t* result_quantization_dimension, int64_t* result_n) {
  if (!valid_quant(q, operand)) return ORC_EINVAL;
  int rc = orc_broadcast_in_dim(operand, operand_data, broadcast_dimensions, result, result_data);
  if (rc != ORC_OK) return rc;
  if (!q->per_axis) {
    *result_quantization_dimension = -1;
    *result_n = 1;
    result_scales[0] = q->scales[0];
    result_zero_points[0] = q->zero_points[0];
    return ORC_OK;
  }
  const int qd = q->quantization_dimension;
  const int rqd = (int)broadcast_dimensions[qd];  // C6
  const int64_t n = result->dims[rqd];
  const bool single = operand->dims[qd] == 1;
  for (int64_t i = 0; i < n; ++i) {
    result_scales[i] = q->scales[single ? 0 : i];
    result_zero_points[i] = q->zero_points[single ? 0 : i];
  }
  *result_quantization_dimension = rqd;
  *result_n = n;
  return ORC_OK;
}

static int64_t prod_dims(const orc_arr* a, int from, int to) {  // dims[from .. to-1]
  int64_t p = 1;
  for (int d = from; d < to; ++d) p *= a->dims[d];
  return p;
}

// reshape: the element at lexicographic position p of the operand goes to lexicographic position p
// of the result (both arrays in their own layouts). result_qdim is the result type's quantization
// dimension (-1 for a per-tensor or unquantized tensor); q may be NULL for an unquantized reshape.
extern "C" int orc_quant_reshape(const orc_arr* operand, const void* operand_data, const orc_quant* q,
                                 const orc_arr* result, int32_t result_qdim, void* result_data) {
  if (!valid_arr(operand) || !valid_arr(result) || operand->dtype != result->dtype) return ORC_EINVAL;
  if (num_elements(operand) != num_elements(result)) return ORC_EINVAL;  // C2
  if (q) {
    if (!valid_quant(q, operand)) return ORC_EINVAL;
    if (q->per_axis) {  // C3
      const int qd = q->quantization_dimension;
      if (result_qdim < 0 || result_qdim >= result->rank) return ORC_EINVAL;
      if (prod_dims(operand, 0, qd) != prod_dims(result, 0, result_qdim)) return ORC_EINVAL;
      if (operand->dims[qd] != result->dims[result_qdim]) return ORC_EINVAL;
      if (prod_dims(operand, qd + 1, operand->rank) != prod_dims(result, result_qdim + 1, result->rank))
        return ORC_EINVAL;
    } else if (result_qdim != -1) {
      return ORC_EINVAL;  // C1: a per-tensor operand stays per-tensor
    }
  }
  int64_t ostride[ORC_MAX_RANK], rstride[ORC_MAX_RANK];
  strides_of(operand, ostride);
  strides_of(result, rstride);
  const int eb = elem_bytes(operand->dtype);
  const int64_t n = num_elements(operand);
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < n; ++p) {
    int64_t oi[ORC_MAX_RANK], ri[ORC_MAX_RANK];
    lex_index(operand->rank, operand->dims, p, oi);
    lex_index(result->rank, result->dims, p, ri);
    int64_t oo = 0, ro = 0;
    for (int d = 0; d < operand->rank; ++d) oo += oi[d] * ostride[d];
    for (int d = 0; d < result->rank; ++d) ro += ri[d] * rstride[d];
    std::memcpy((char*)result_data + ro * eb, (const char*)operand_data + oo * eb, eb);
  }
  return ORC_OK;
}

// ----------------------------------------------------------------------------------------------
// Quantized elementwise binary ops ("StableHLO Specification", sections add, divide, maximum,
// minimum, multiply: dequantize_op_quantize(op, lhs, rhs, type(result))): both operands dequantized,
// the op in IEEE f32 (maximum / minimum: NaN propagates, -0 < +0), the result quantized with the
// result's parameters. Operands and result share dims; each has its own layout. op: 0 add, 1 divide,
// 2 maximum, 3 minimum, 4 multiply.
// ----------------------------------------------------------------------------------------------
static float ieee_binary(int op, float a, float b) {
  switch (op) {
    case 0: return a + b;
    case 1: return a / b;
    case 2:
    case 3: {
      if (std::isnan(a) || std::isnan(b)) return NAN;
      if (a == b) {  // equal values, possibly zeros of different sign: maximum(-0, +0) = +0
        bool neg_a = std::signbit(a), neg_b = std::signbit(b);
        if (op == 2) return neg_a ? b : a;
        return neg_a ? a : b;
      }
      return op == 2 ? (a > b ? a : b) : (a < b ? a : b);
    }
    default: return a * b;
  }
}

extern "C" int orc_quant_binary(int op, const orc_arr* lhs, const void* l_data, const orc_quant* lq,
                                const orc_arr* rhs, const void* r_data, const orc_quant* rq, const orc_arr* out,
                                void* out_data, const orc_quant* oq) {
  if (op < 0 || op > 4) return ORC_EINVAL;
  if (!valid_arr(lhs) || !valid_arr(rhs) || !valid_arr(out)) return ORC_EINVAL;
  if (rhs->rank != lhs->rank || out->rank != lhs->rank) return ORC_EINVAL;
  for (int d = 0; d < lhs->rank; ++d)
    if (rhs->dims[d] != lhs->dims[d] || out->dims[d] != lhs->dims[d]) return ORC_EINVAL;
  if (!valid_quant(lq, lhs) || !valid_quant(rq, rhs) || !valid_quant(oq, out)) return ORC_EINVAL;
  if (lq->per_axis || rq->per_axis || oq->per_axis) return ORC_EINVAL;  // per-tensor operands (I1, I2)
  int64_t ls[ORC_MAX_RANK], rs[ORC_MAX_RANK], os[ORC_MAX_RANK];
  strides_of(lhs, ls);
  strides_of(rhs, rs);
  strides_of(out, os);
  const int64_t n = num_elements(lhs);
#pragma omp parallel for schedule(static)
  for (int64_t e = 0; e < n; ++e) {
    int64_t idx[ORC_MAX_RANK];
    lex_index(lhs->rank, lhs->dims, e, idx);
    int64_t lo = 0, ro = 0, oo = 0;
    for (int d = 0; d < lhs->rank; ++d) { lo += idx[d] * ls[d]; ro += idx[d] * rs[d]; oo += idx[d] * os[d]; }
    const float a = dequantize_one(lq, (int32_t)load_elem(l_data, lhs->dtype, lo), idx);
    const float b = dequantize_one(rq, (int32_t)load_elem(r_data, rhs->dtype, ro), idx);
    store_elem(out_data, out->dtype, oo, (double)quantize_one(oq, ieee_binary(op, a, b), idx));
  }
  return ORC_OK;
}

// ----------------------------------------------------------------------------------------------
// Scalar entry points used to pin the elementwise rules.
// ----------------------------------------------------------------------------------------------
extern "C" double orc_round_to(double v, int dtype) { return round_to<double>(v, dtype); }
extern "C" double orc_exp(double x, int dtype) { return cr_exp(round_to<double>(x, dtype), dtype); }
extern "C" double orc_log(double x, int dtype) { return cr_log(round_to<double>(x, dtype), dtype); }
extern "C" double orc_maximum(double a, double b) { return (double)ieee_maximum(a, b); }
extern "C" int orc_quantize(const orc_quant* q, float real, const int64_t* idx) { return quantize_one(q, real, idx); }
extern "C" float orc_dequantize(const orc_quant* q, int32_t code, const int64_t* idx) { return dequantize_one(q, code, idx); }

// Exhaustive check helper: for count consecutive f32 bit patterns starting at first_bits, compares
// cand[i] (bit pattern of a claimed correctly rounded f32 log) with the oracle's value. NaN results
// match any NaN pattern. Returns the number of mismatches; the first max_report mismatching input
// patterns (in ascending order) are written to report.
// Counts the candidates (f32 bit patterns of f(x) for the consecutive inputs x starting at first_bits)
// that differ from the oracle's correctly rounded f32 value; any NaN matches a NaN.
template <double (*F)(double, int)>
static int64_t check_f32(uint32_t first_bits, int64_t count, const uint32_t* cand, uint32_t* report,
                         int64_t max_report) {
  std::vector<uint8_t> bad_flag((size_t)count, 0);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) {
    uint32_t b = first_bits + (uint32_t)i;
    float x; std::memcpy(&x, &b, 4);
    float y = (float)F(x, ORC_F32);
    uint32_t yb; std::memcpy(&yb, &y, 4);
    bool cand_nan = (cand[i] & 0x7F800000u) == 0x7F800000u && (cand[i] & 0x7FFFFFu) != 0;
    bool same = std::isnan(y) ? cand_nan : yb == cand[i];
    bad_flag[(size_t)i] = same ? 0 : 1;
  }
  int64_t bad = 0;
  for (int64_t i = 0; i < count; ++i) {
    if (!bad_flag[(size_t)i]) continue;
    if (bad < max_report) report[bad] = first_bits + (uint32_t)i;
    ++bad;
  }
  return bad;
}

extern "C" int64_t orc_check_log_f32(uint32_t first_bits, int64_t count, const uint32_t* cand,
                                     uint32_t* report, int64_t max_report) {
  return check_f32<cr_log>(first_bits, count, cand, report, max_report);
}

extern "C" int64_t orc_check_tanh_f32(uint32_t first_bits, int64_t count, const uint32_t* cand,
                                      uint32_t* report, int64_t max_report) {
  return check_f32<cr_tanh>(first_bits, count, cand, report, max_report);
}

extern "C" int64_t orc_check_exp_f32(uint32_t first_bits, int64_t count, const uint32_t* cand,
                                     uint32_t* report, int64_t max_report) {
  return check_f32<cr_exp>(first_bits, count, cand, report, max_report);
}

extern "C" void orc_set_num_threads(int n) {
#ifdef _OPENMP
  omp_set_num_threads(n);
#else
  (void)n;
#endif
}

extern "C" int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

