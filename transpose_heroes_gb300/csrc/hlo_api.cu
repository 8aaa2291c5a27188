// C-ABI entry points of libhlofusion: argument validation against the spec's constraints, layout
// canonicalization (unit dimensions dropped, dimensions adjacent in both memory orders merged), plan
// selection and kernel launch. No device memory is allocated here.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "hlo_fusion.h"
#include "hlo_internal.h"

using namespace hlo;

namespace {

thread_local std::string g_err;

hlo_status fail(hlo_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

hlo_status ok() {
  g_err.clear();
  return HLO_OK;
}

hlo_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(HLO_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool is_float(int dt) { return dt == F32 || dt == BF16 || dt == F16; }

// ---- arrays --------------------------------------------------------------------------------------
hlo_status check_array(const hlo_array* a, const char* what) {
  if (!a) return fail(HLO_ERR_INVALID_ARG, "%s: array descriptor is NULL", what);
  if (a->rank < 0 || a->rank > HLO_MAX_RANK)
    return fail(HLO_ERR_INVALID_ARG, "%s: rank %d outside 0..%d", what, a->rank, HLO_MAX_RANK);
  if (dt_bytes(a->dtype) == 0) return fail(HLO_ERR_INVALID_ARG, "%s: unknown element type %d", what, a->dtype);
  bool seen[HLO_MAX_RANK] = {false};
  for (int k = 0; k < a->rank; ++k) {
    if (a->dims[k] < 0) return fail(HLO_ERR_INVALID_ARG, "%s: dimension %d has negative size", what, k);
    const int64_t d = a->minor_to_major[k];
    if (d < 0 || d >= a->rank || seen[d])
      return fail(HLO_ERR_INVALID_ARG, "%s: minor_to_major is not a permutation of 0..%d", what, a->rank - 1);
    seen[d] = true;
  }
  // element count must fit comfortably in 62 bits of bytes
  long double n = 1;
  for (int k = 0; k < a->rank; ++k) n *= (long double)a->dims[k];
  if (n * dt_bytes(a->dtype) > 4.0e18L) return fail(HLO_ERR_INVALID_ARG, "%s: array too large", what);
  return HLO_OK;
}

int64_t numel(const hlo_array& a) {
  int64_t n = 1;
  for (int k = 0; k < a.rank; ++k) n *= a.dims[k];
  return n;
}

// stride[d] of logical dimension d in elements, from minor_to_major.
void strides_of(const hlo_array& a, int64_t* stride) {
  int64_t s = 1;
  for (int k = 0; k < a.rank; ++k) {
    stride[a.minor_to_major[k]] = s;
    s *= a.dims[a.minor_to_major[k]];
  }
}

bool ranges_overlap(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
  if (abytes <= 0 || bbytes <= 0) return false;
  const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + (uintptr_t)bbytes && b0 < a0 + (uintptr_t)abytes;
}

// ---- chains --------------------------------------------------------------------------------------
// A constant of the chain as a value of float element type dt: round to nearest, ties to even, at the
// type's precision (8 significand bits for bf16, 11 for f16, 24 for f32), with gradual underflow and
// overflow to infinity ("StableHLO Specification", section "constant": the literal is a value of the
// element type).
static float constant_of_type(double v, int dt) {
  if (v == 0 || std::isnan(v) || std::isinf(v)) return (float)v;
  const int prec = dt == BF16 ? 8 : dt == F16 ? 11 : 24;
  const int emin = dt == F16 ? -14 : -126, emax = dt == F16 ? 15 : 127;
  int e;
  std::frexp(v, &e);
  const int lead = std::max(e - 1, emin);
  const double quantum = std::ldexp(1.0, lead - prec + 1);
  const double r = std::nearbyint(v / quantum) * quantum;  // v / quantum is exact
  const double maxv = std::ldexp(1.0, emax) * (2.0 - std::ldexp(1.0, 1 - prec));
  if (std::fabs(r) > maxv) return v > 0 ? INFINITY : -INFINITY;
  return (float)r;  // exact: r has at most prec <= 24 significand bits
}

// Validates a chain attached to array `arr` and builds the kernel descriptor.
hlo_status make_chain(const hlo_ew_chain* c, const hlo_array& arr, bool allow_bcast, const char* what, Chain* out,
                      int force_dt = -1) {
  std::memset(out, 0, sizeof *out);
  out->dt = force_dt >= 0 ? force_dt : arr.dtype;
  if (!c || c->n_ops == 0) return HLO_OK;
  if (c->n_ops < 0 || c->n_ops > HLO_MAX_EW_OPS)
    return fail(HLO_ERR_INVALID_ARG, "%s: n_ops %d outside 0..%d", what, c->n_ops, HLO_MAX_EW_OPS);
  if (!is_float(out->dt))
    return fail(HLO_ERR_INVALID_ARG, "%s: elementwise ops need a floating-point element type (exponential/log C1)", what);
  out->n = c->n_ops;
  out->round16 = c->round_intermediates ? 1 : 0;
  for (int k = 0; k < c->n_ops; ++k) {
    const int op = c->ops[k];
    if (op < HLO_EW_EXP || op > HLO_EW_MUL_INPUT) return fail(HLO_ERR_INVALID_ARG, "%s: unknown op %d", what, op);
    out->op[k] = op;
    if (op == HLO_EW_ADD_CONST || op == HLO_EW_MUL_CONST) out->imm[k] = constant_of_type(c->imm[k], out->dt);
    if (op != HLO_EW_ADD_BCAST) continue;
    if (!allow_bcast) return fail(HLO_ERR_UNSUPPORTED, "%s: add of a broadcast operand is not supported here", what);
    hlo_status st = check_array(&c->bcast, "broadcast operand");
    if (st != HLO_OK) return st;
    const hlo_array& b = c->bcast;
    if (b.dtype != out->dt)
      return fail(HLO_ERR_INVALID_ARG, "%s: add (C1): broadcast operand type %d differs from %d", what, b.dtype, out->dt);
    bool used[HLO_MAX_RANK] = {false};
    int64_t bstr[HLO_MAX_RANK];
    strides_of(b, bstr);
    for (int d = 0; d < b.rank; ++d) {
      const int64_t bd = c->bcast_dimensions[d];
      if (bd < 0 || bd >= arr.rank)
        return fail(HLO_ERR_INVALID_ARG, "%s: broadcast_in_dim (C3): broadcast_dimensions[%d] = %lld out of range",
                    what, d, (long long)bd);
      if (used[bd]) return fail(HLO_ERR_INVALID_ARG, "%s: broadcast_in_dim (C4): broadcast_dimensions not unique", what);
      used[bd] = true;
      if (b.dims[d] != 1 && b.dims[d] != arr.dims[bd])
        return fail(HLO_ERR_INVALID_ARG, "%s: broadcast_in_dim (C5): operand dim %d has size %lld, result dim %lld has %lld",
                    what, d, (long long)b.dims[d], (long long)bd, (long long)arr.dims[bd]);
      if (b.dims[d] != 1) out->bstride[bd] += bstr[d];
    }
    if (!c->bcast_ptr && numel(b) > 0) return fail(HLO_ERR_INVALID_ARG, "%s: broadcast operand pointer is NULL", what);
    out->bptr = c->bcast_ptr;
    out->bdt = b.dtype;
  }
  return HLO_OK;
}

bool chain_has_bcast(const Chain& c) {
  for (int k = 0; k < c.n; ++k)
    if (c.op[k] == OP_ADD_BCAST) return true;
  return false;
}

// Builds an IndexMap over axes (major first) with the given sizes and target strides, merging axes
// that are contiguous in the target.
IndexMap make_map(const std::vector<int64_t>& size, const std::vector<int64_t>& stride) {
  std::vector<int64_t> sz, st;
  for (size_t j = 0; j < size.size(); ++j) {
    if (size[j] == 1) continue;
    if (!sz.empty() && st.back() == stride[j] * size[j]) {
      sz.back() *= size[j];
      st.back() = stride[j];
    } else {
      sz.push_back(size[j]);
      st.push_back(stride[j]);
    }
  }
  IndexMap m;
  std::memset(&m, 0, sizeof m);
  m.n = (int)sz.size();
  for (int j = 0; j < m.n; ++j) {
    m.size[j] = sz[j];
    m.stride[j] = st[j];
  }
  m.identity = (m.n == 0 || (m.n == 1 && st[0] == 1)) ? 1 : 0;
  return m;
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Host-side fault injection, for tests of the error path that fault no GPU: when the environment
// variable HLOFUSION_FAULT names an entry point (or is "all"), that entry point validates its arguments
// as usual and then returns HLO_ERR_CUDA with an "injected fault" message before it enqueues anything.
// The variable is read on every call; unset, it costs one getenv.
bool injected(const char* site) {
  const char* v = std::getenv("HLOFUSION_FAULT");
  return v && *v && (std::strcmp(v, "all") == 0 || std::strcmp(v, site) == 0);
}
#define HLO_INJECT(site) \
  if (injected(site)) return fail(HLO_ERR_CUDA, "%s: injected fault (HLOFUSION_FAULT)", site)

// Rows and row length of a reduce whose reduced dimensions are the minor-most physical ones (unit
// dimensions dropped); false for any other pattern.
bool row_geometry(const hlo_array& in, const bool* red, int64_t* rows, int64_t* len) {
  int64_t r = 1, l = 1;
  bool in_reduced_tail = true;  // walking from the minor end
  for (int k = 0; k < in.rank; ++k) {
    const int d = (int)in.minor_to_major[k];
    if (in.dims[d] == 1) continue;
    if (red[d]) {
      if (!in_reduced_tail) return false;
      l *= in.dims[d];
    } else {
      in_reduced_tail = false;
      r *= in.dims[d];
    }
  }
  *rows = r;
  *len = l;
  return true;
}

// ---- quantization parameters ---------------------------------------------------------------------
hlo_status check_quant(const hlo_quant* q, const hlo_array& a, const char* what, QuantParams* out) {
  std::memset(out, 0, sizeof *out);
  if (!q) return fail(HLO_ERR_INVALID_ARG, "%s: quantization parameters are NULL", what);
  const int qd = q->quantization_dimension;
  if (qd < -1 || qd >= a.rank)
    return fail(HLO_ERR_INVALID_ARG, "%s: quantized type (C12): quantization_dimension %d out of range", what, qd);
  if (qd < 0 && q->n != 1)
    return fail(HLO_ERR_INVALID_ARG, "%s: quantized type (C11): per-tensor quantization needs exactly 1 scale", what);
  if (qd >= 0 && q->n != a.dims[qd])
    return fail(HLO_ERR_INVALID_ARG, "%s: quantized type (C13): %lld scales for a dimension of size %lld", what,
                (long long)q->n, (long long)a.dims[qd]);
  if (!(-128 <= q->storage_min && q->storage_min < q->storage_max && q->storage_max <= 127))
    return fail(HLO_ERR_INVALID_ARG, "%s: quantized type (C4): storage range [%d, %d] invalid for i8", what,
                q->storage_min, q->storage_max);
  if (q->host_scales) {
    for (int64_t i = 0; i < q->n; ++i) {
      const float s = q->host_scales[i];
      if (!(s > 0.0f)) return fail(HLO_ERR_INVALID_ARG, "%s: quantized type (C6): scale[%lld] is not > 0", what, (long long)i);
      if (!std::isfinite(s)) return fail(HLO_ERR_INVALID_ARG, "%s: quantized type (C7): scale[%lld] is not finite", what, (long long)i);
    }
  }
  if (q->host_zero_points) {
    for (int64_t i = 0; i < q->n; ++i) {
      const int32_t z = q->host_zero_points[i];
      if (z < q->storage_min || z > q->storage_max)
        return fail(HLO_ERR_INVALID_ARG, "%s: quantized type (C8): zero_point[%lld] = %d outside [%d, %d]", what,
                    (long long)i, z, q->storage_min, q->storage_max);
    }
  }
  out->axis = qd;
  out->smin = q->storage_min;
  out->smax = q->storage_max;
  out->max_abs_scale = -1.0f;
  if (q->host_scales) {
    float m = 0.0f;
    for (int64_t i = 0; i < q->n; ++i) m = std::max(m, std::fabs(q->host_scales[i]));
    out->max_abs_scale = m;
  }
  if (qd < 0) {
    if (!q->host_scales || !q->host_zero_points)
      return fail(HLO_ERR_INVALID_ARG, "%s: per-tensor parameters need host_scales and host_zero_points", what);
    out->scale = q->host_scales[0];
    out->zp = q->host_zero_points[0];
    volatile float one = 1.0f;
    out->inv_scale = one / out->scale;  // IEEE division on the host: RN(1/scale)
  } else {
    if ((!q->scales || !q->zero_points) && q->n > 0)
      return fail(HLO_ERR_INVALID_ARG, "%s: per-axis parameters need device scales and zero_points", what);
    out->scales = q->scales;
    out->zps = q->zero_points;
  }
  return HLO_OK;
}

// ---- physical canonicalization of a permutation ---------------------------------------------------
// Input logical dims in input physical order (major first) and, for the output, the input logical dim
// each output physical axis reads. Unit dims are dropped; runs adjacent in both orders are merged.
struct Canon {
  int k = 0;
  int64_t size[HLO_MAX_RANK];
  int out_pos[HLO_MAX_RANK];  // position of canonical axis j in the output physical order (major first)
};

Canon canonicalize(const hlo_array& in, const int64_t* perm, const int64_t* out_m2m) {
  const int rank = in.rank;
  std::vector<int> pin, pout;  // input logical dims, major first
  for (int k = rank - 1; k >= 0; --k)
    if (in.dims[in.minor_to_major[k]] != 1) pin.push_back((int)in.minor_to_major[k]);
  for (int k = rank - 1; k >= 0; --k) {
    const int od = (int)out_m2m[k];
    const int idim = (int)perm[od];
    if (in.dims[idim] != 1) pout.push_back(idim);
  }
  // groups: maximal runs of pin that also appear consecutively, in the same order, in pout
  std::vector<std::vector<int>> groups;
  for (size_t i = 0; i < pin.size(); ++i) {
    if (!groups.empty()) {
      const int prev = groups.back().back();
      const auto itp = std::find(pout.begin(), pout.end(), prev);
      if (itp + 1 != pout.end() && *(itp + 1) == pin[i]) {
        groups.back().push_back(pin[i]);
        continue;
      }
    }
    groups.push_back({pin[i]});
  }
  Canon c;
  c.k = (int)groups.size();
  for (int j = 0; j < c.k; ++j) {
    int64_t s = 1;
    for (int d : groups[j]) s *= in.dims[d];
    c.size[j] = s;
    const int first = groups[j].front();
    int pos = 0;
    for (int g = 0; g < c.k; ++g) {
      // rank of group j among groups by the output position of their first dims
      const int fg = groups[g].front();
      const auto pj = std::find(pout.begin(), pout.end(), first) - pout.begin();
      const auto pg = std::find(pout.begin(), pout.end(), fg) - pout.begin();
      if (pg < pj) ++pos;
    }
    c.out_pos[j] = pos;
  }
  return c;
}

// ---- planners --------------------------------------------------------------------------------------
hlo_status plan_gather_plain(const hlo_array& in, const void* in_ptr, const hlo_array& out, void* out_ptr,
                             const int64_t* perm, int self_add, const Chain& pro, const Chain& epi, cudaStream_t s) {
  GatherPlan g;
  std::memset(&g, 0, sizeof g);
  g.in = in_ptr;
  g.out = out_ptr;
  g.kind = G_PLAIN;
  g.rank = out.rank;
  g.n = numel(out);
  int64_t istr[HLO_MAX_RANK];
  strides_of(in, istr);
  for (int j = 0; j < out.rank; ++j) {
    const int od = (int)out.minor_to_major[out.rank - 1 - j];
    g.out_size[j] = out.dims[od];
    g.out_logical[j] = od;
  }
  for (int k = 0; k < out.rank; ++k) {
    g.perm[k] = (int)perm[k];
    g.in_stride_of_out[k] = istr[perm[k]];
    g.self_stride_of_out[k] = istr[k];
  }
  g.self_add = self_add;
  g.in_dt = in.dtype;
  g.out_dt = out.dtype;
  g.elem_bytes = dt_bytes(in.dtype);
  g.pro = pro;
  g.epi = epi;
  return cuda_status(launch_gather(g, s), "gather kernel launch");
}

}  // namespace

// The occupancy queries below may leave an error of their own in CUDA's sticky last-error slot; that
// one is cleared so the next launch check does not report it. An error that was already pending when
// the query began (from the caller's earlier asynchronous work) is left in place.
static void clear_query_error(cudaError_t pending) {
  if (pending == cudaSuccess) cudaGetLastError();
}

int hlo::device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

void hlo::table_cluster_shape(const void* kernel, int threads, size_t smem, int* cluster_size, int* clusters) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, std::pair<int, int>> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_pair(kernel, dev);
  auto it = cache.find(key);
  if (it == cache.end()) {
    const cudaError_t pending = cudaPeekAtLastError();
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    std::pair<int, int> best(2, 1);
    for (int cs : {8, 4, 2}) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = cs;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(cs, 1, 1);
      cfg.blockDim = dim3(threads, 1, 1);
      cfg.dynamicSmemBytes = smem;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) n = 0;
      if (n >= 1) {  // the largest size that fits: building the table costs 65536 / size evaluations per block
        best = std::make_pair(cs, n);
        break;
      }
    }
    clear_query_error(pending);
    it = cache.emplace(key, best).first;
  }
  *cluster_size = it->second.first;
  *clusters = it->second.second;
}

int hlo::kernel_blocks_per_sm(const void* kernel, int threads, size_t smem) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_pair(kernel, dev * 4096 + threads);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  const cudaError_t pending = cudaPeekAtLastError();
  if (smem > 0) cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, threads, smem) != cudaSuccess || nb < 1) nb = 1;
  clear_query_error(pending);
  cache[key] = nb;
  return nb;
}

namespace hlo {
namespace {
std::vector<FaultReader>& fault_readers() {
  static std::vector<FaultReader> readers;  // filled while the library's units are initialised
  return readers;
}
}  // namespace

int register_fault_reader(FaultReader r) {
  fault_readers().push_back(r);
  return static_cast<int>(fault_readers().size()) - 1;
}

cudaError_t read_all_faults(unsigned int* faults, bool clear) {
  *faults = 0;
  for (FaultReader r : fault_readers()) {
    unsigned int f = 0;
    const cudaError_t e = r(&f, clear);
    if (e != cudaSuccess) return e;
    *faults |= f;
  }
  return cudaSuccess;
}
}  // namespace hlo

extern "C" {

// ---- quantized elementwise binary ops ------------------------------------------------------------------
hlo_status hlo_quant_binary(int32_t op, const hlo_array* lhs, const void* lhs_ptr, const hlo_quant* lhs_q,
                            const hlo_array* rhs, const void* rhs_ptr, const hlo_quant* rhs_q, const hlo_array* out,
                            void* out_ptr, const hlo_quant* out_q, void* stream) {
  if (op < HLO_QOP_ADD || op > HLO_QOP_MULTIPLY) return fail(HLO_ERR_INVALID_ARG, "quantized op: unknown op %d", op);
  hlo_status st;
  const hlo_array* arrs[3] = {lhs, rhs, out};
  const char* names[3] = {"quantized lhs", "quantized rhs", "quantized result"};
  for (int a = 0; a < 3; ++a) {
    if ((st = check_array(arrs[a], names[a])) != HLO_OK) return st;
    if (arrs[a]->dtype != HLO_S8) return fail(HLO_ERR_UNSUPPORTED, "%s: storage type must be s8", names[a]);
  }
  for (int a = 1; a < 3; ++a) {
    if (arrs[a]->rank != lhs->rank) return fail(HLO_ERR_INVALID_ARG, "%s (C1): rank differs from lhs", names[a]);
    for (int d = 0; d < lhs->rank; ++d)
      if (arrs[a]->dims[d] != lhs->dims[d]) return fail(HLO_ERR_INVALID_ARG, "%s (C1): shape differs from lhs", names[a]);
  }
  QuantBinaryPlan p;
  std::memset(&p, 0, sizeof p);
  const hlo_quant* qs[3] = {lhs_q, rhs_q, out_q};
  QuantParams* qp[3] = {&p.ql, &p.qr, &p.qo};
  for (int a = 0; a < 3; ++a) {
    if ((st = check_quant(qs[a], *arrs[a], names[a], qp[a])) != HLO_OK) return st;
    if (qp[a]->axis >= 0)
      return fail(HLO_ERR_INVALID_ARG, "%s (I1, I2): per-tensor quantized tensors only", names[a]);
  }
  const int64_t n = numel(*lhs);
  if (n > 0 && (!lhs_ptr || !rhs_ptr || !out_ptr)) return fail(HLO_ERR_INVALID_ARG, "quantized op: NULL pointer");
  if (ranges_overlap(out_ptr, n, lhs_ptr, n) || ranges_overlap(out_ptr, n, rhs_ptr, n))
    return fail(HLO_ERR_INVALID_ARG, "quantized op: the result overlaps an operand");
  if (n == 0) return ok();
  p.lhs = static_cast<const int8_t*>(lhs_ptr);
  p.rhs = static_cast<const int8_t*>(rhs_ptr);
  p.out = static_cast<int8_t*>(out_ptr);
  p.n = n;
  p.op = op;
  bool same_layout = true;
  for (int a = 1; a < 3; ++a)
    for (int d = 0; d < lhs->rank; ++d) same_layout = same_layout && arrs[a]->minor_to_major[d] == lhs->minor_to_major[d];
  if (same_layout) {  // the same physical offset holds the same logical index in all three
    p.lmap = p.rmap = p.omap = make_map({n}, {1});
  } else {
    std::vector<int64_t> sz(lhs->dims, lhs->dims + lhs->rank);
    IndexMap* maps[3] = {&p.lmap, &p.rmap, &p.omap};
    for (int a = 0; a < 3; ++a) {
      int64_t str[HLO_MAX_RANK];
      strides_of(*arrs[a], str);
      *maps[a] = make_map(sz, std::vector<int64_t>(str, str + lhs->rank));
    }
  }
  HLO_INJECT("hlo_quant_binary");
  return cuda_status(launch_quant_binary(p, as_stream(stream)), "quantized op launch");
}

// ---- variadic reduce: max / argmax ------------------------------------------------------------------
hlo_status hlo_reduce_max_argmax(const hlo_array* in, const void* in_ptr, const hlo_array* idx, const void* idx_ptr,
                                 const int64_t* dimensions, int32_t n_dimensions, double init_value,
                                 int64_t init_index, const hlo_array* out, void* out_ptr, const hlo_array* out_idx,
                                 void* out_idx_ptr, void* stream) {
  hlo_status st = check_array(in, "argmax input");
  if (st != HLO_OK) return st;
  if ((st = check_array(out, "argmax values")) != HLO_OK) return st;
  if ((st = check_array(out_idx, "argmax indices")) != HLO_OK) return st;
  if (!is_float(in->dtype)) return fail(HLO_ERR_UNSUPPORTED, "argmax: input element type %d not supported", in->dtype);
  if (out->dtype != in->dtype)
    return fail(HLO_ERR_INVALID_ARG, "variadic reduce (C7): values type %d differs from input %d", out->dtype, in->dtype);
  if (out_idx->dtype != HLO_S32) return fail(HLO_ERR_UNSUPPORTED, "argmax: indices must be s32");
  if (init_index < INT32_MIN || init_index > INT32_MAX) return fail(HLO_ERR_INVALID_ARG, "argmax: init_index outside s32");
  if (n_dimensions < 0 || n_dimensions > in->rank)
    return fail(HLO_ERR_INVALID_ARG, "reduce (C4): %d dimensions for rank %d", n_dimensions, in->rank);
  if (n_dimensions > 0 && !dimensions) return fail(HLO_ERR_INVALID_ARG, "argmax: dimensions is NULL");
  bool red[HLO_MAX_RANK] = {false};
  for (int i = 0; i < n_dimensions; ++i) {
    const int64_t d = dimensions[i];
    if (d < 0 || d >= in->rank)
      return fail(HLO_ERR_INVALID_ARG, "reduce (C4): dimension %lld outside [0, %d)", (long long)d, in->rank);
    if (red[d]) return fail(HLO_ERR_INVALID_ARG, "reduce (C5): dimension %lld repeated", (long long)d);
    red[d] = true;
  }
  if (idx_ptr) {
    if (!idx) return fail(HLO_ERR_INVALID_ARG, "argmax: index array descriptor is NULL");
    if ((st = check_array(idx, "argmax index input")) != HLO_OK) return st;
    if (idx->dtype != HLO_S32) return fail(HLO_ERR_UNSUPPORTED, "argmax: index input must be s32");
    if (idx->rank != in->rank) return fail(HLO_ERR_INVALID_ARG, "variadic reduce (C2): index input rank differs");
    for (int d = 0; d < in->rank; ++d)
      if (idx->dims[d] != in->dims[d]) return fail(HLO_ERR_INVALID_ARG, "variadic reduce (C2): index input shape differs");
  } else if (n_dimensions != 1) {
    return fail(HLO_ERR_INVALID_ARG, "argmax: without an index input exactly one dimension is reduced");
  }
  std::vector<int> kept, redd;
  for (int d = 0; d < in->rank; ++d) (red[d] ? redd : kept).push_back(d);
  for (const hlo_array* o : {out, out_idx}) {
    if (o->rank != (int)kept.size())
      return fail(HLO_ERR_INVALID_ARG, "reduce (C7): output rank %d, expected %d", o->rank, (int)kept.size());
    for (size_t k = 0; k < kept.size(); ++k)
      if (o->dims[k] != in->dims[kept[k]])
        return fail(HLO_ERR_INVALID_ARG, "reduce (C7): output dim %d is %lld, expected %lld", (int)k,
                    (long long)o->dims[k], (long long)in->dims[kept[k]]);
  }
  const int64_t n_in = numel(*in), n_out = numel(*out);
  if (n_in > 0 && !in_ptr) return fail(HLO_ERR_INVALID_ARG, "argmax: input pointer is NULL");
  if (n_out > 0 && (!out_ptr || !out_idx_ptr)) return fail(HLO_ERR_INVALID_ARG, "argmax: output pointer is NULL");
  const int64_t vb = n_out * dt_bytes(out->dtype), ib = n_out * 4;
  if (ranges_overlap(in_ptr, n_in * dt_bytes(in->dtype), out_ptr, vb) ||
      ranges_overlap(in_ptr, n_in * dt_bytes(in->dtype), out_idx_ptr, ib) || ranges_overlap(out_ptr, vb, out_idx_ptr, ib) ||
      (idx_ptr && (ranges_overlap(idx_ptr, n_in * 4, out_ptr, vb) || ranges_overlap(idx_ptr, n_in * 4, out_idx_ptr, ib))))
    return fail(HLO_ERR_INVALID_ARG, "argmax: an output overlaps another buffer");
  if (n_out == 0) return ok();
  int64_t vstr[HLO_MAX_RANK], kstr[HLO_MAX_RANK] = {0}, ostr[HLO_MAX_RANK], istr[HLO_MAX_RANK];
  strides_of(*in, vstr);
  if (idx_ptr) strides_of(*idx, kstr);
  strides_of(*out, ostr);
  strides_of(*out_idx, istr);
  // kept dims walked lexicographically (output linear index), reduced dims likewise (walk position)
  std::vector<int64_t> ksz, kv, kk, ko, ki, rsz, rv, rk;
  for (size_t k = 0; k < kept.size(); ++k) {
    ksz.push_back(in->dims[kept[k]]);
    kv.push_back(vstr[kept[k]]);
    kk.push_back(kstr[kept[k]]);
    ko.push_back(ostr[k]);
    ki.push_back(istr[k]);
  }
  for (int d : redd) {
    rsz.push_back(in->dims[d]);
    rv.push_back(vstr[d]);
    rk.push_back(kstr[d]);
  }
  ArgmaxPlan p;
  std::memset(&p, 0, sizeof p);
  p.v = in_ptr;
  p.k = static_cast<const int32_t*>(idx_ptr);
  p.out = out_ptr;
  p.out_idx = static_cast<int32_t*>(out_idx_ptr);
  p.dt = in->dtype;
  p.n_out = n_out;
  p.n_red = 1;
  for (int64_t r : rsz) p.n_red *= r;
  p.vkept = make_map(ksz, kv);
  p.kkept = make_map(ksz, kk);
  p.okept = make_map(ksz, ko);
  p.ikept = make_map(ksz, ki);
  p.vred = make_map(rsz, rv);
  p.kred = make_map(rsz, rk);
  p.init_value = constant_of_type(init_value, in->dtype);
  p.init_index = (int32_t)init_index;
  HLO_INJECT("hlo_reduce_max_argmax");
  return cuda_status(launch_argmax(p, as_stream(stream)), "argmax launch");
}

// ---- quantized data movement: broadcast_in_dim and reshape -------------------------------------------
hlo_status hlo_quant_broadcast_in_dim(const hlo_array* operand, const void* operand_ptr, const hlo_quant* operand_q,
                                      const int64_t* broadcast_dimensions, const hlo_array* result, void* result_ptr,
                                      float* result_scales, int32_t* result_zero_points,
                                      int32_t* result_quantization_dimension, void* stream) {
  hlo_status st = check_array(operand, "broadcast_in_dim operand");
  if (st != HLO_OK) return st;
  if ((st = check_array(result, "broadcast_in_dim result")) != HLO_OK) return st;
  if (operand->dtype != S8 || result->dtype != S8)
    return fail(HLO_ERR_UNSUPPORTED, "quantized broadcast_in_dim: storage type must be s8 for operand and result");
  QuantParams qp;
  if ((st = check_quant(operand_q, *operand, "broadcast_in_dim operand", &qp)) != HLO_OK) return st;
  if (operand->rank > 0 && !broadcast_dimensions)
    return fail(HLO_ERR_INVALID_ARG, "broadcast_in_dim (C2): broadcast_dimensions is NULL");
  bool used[HLO_MAX_RANK] = {false};
  for (int d = 0; d < operand->rank; ++d) {
    const int64_t bd = broadcast_dimensions[d];
    if (bd < 0 || bd >= result->rank)
      return fail(HLO_ERR_INVALID_ARG, "broadcast_in_dim (C3): broadcast_dimensions[%d] = %lld out of range", d,
                  (long long)bd);
    if (used[bd]) return fail(HLO_ERR_INVALID_ARG, "broadcast_in_dim (C4): broadcast_dimensions not unique");
    used[bd] = true;
    if (operand->dims[d] != 1 && operand->dims[d] != result->dims[bd])
      return fail(HLO_ERR_INVALID_ARG, "broadcast_in_dim (C5): operand dim %d has size %lld, result dim %lld has %lld", d,
                  (long long)operand->dims[d], (long long)bd, (long long)result->dims[bd]);
  }
  if (!result_quantization_dimension)
    return fail(HLO_ERR_INVALID_ARG, "quantized broadcast_in_dim: result_quantization_dimension is NULL");
  // C1, C6: the result's quantization dimension and the number of its (scale, zero_point) pairs
  const int rqd = qp.axis < 0 ? -1 : (int)broadcast_dimensions[qp.axis];
  const int64_t n_params = rqd < 0 ? 1 : result->dims[rqd];
  if (n_params > 0 && (!result_scales || !result_zero_points))
    return fail(HLO_ERR_INVALID_ARG, "quantized broadcast_in_dim: result parameter buffers are NULL");
  const int64_t n_in = numel(*operand), n_out = numel(*result);
  if (n_out > 0 && (!result_ptr || (n_in > 0 && !operand_ptr)))
    return fail(HLO_ERR_INVALID_ARG, "quantized broadcast_in_dim: NULL data pointer");
  if (ranges_overlap(operand_ptr, n_in, result_ptr, n_out) ||
      ranges_overlap(result_scales, n_params * 4, result_ptr, n_out) ||
      ranges_overlap(result_zero_points, n_params * 4, result_ptr, n_out) ||
      ranges_overlap(result_scales, n_params * 4, result_zero_points, n_params * 4))
    return fail(HLO_ERR_INVALID_ARG, "quantized broadcast_in_dim: output buffers overlap an input or each other");
  HLO_INJECT("hlo_quant_broadcast_in_dim");
  const cudaStream_t s = as_stream(stream);
  *result_quantization_dimension = rqd;
  cudaError_t e = rqd < 0 ? launch_quant_params(nullptr, nullptr, qp.scale, qp.zp, 1, result_scales,
                                                result_zero_points, 1, s)
                          : launch_quant_params(qp.scales, qp.zps, 0.f, 0, operand->dims[qp.axis] == 1 ? 1 : 0,
                                                result_scales, result_zero_points, n_params, s);
  if (e != cudaSuccess) return cuda_status(e, "quantized parameter kernel launch");
  if (n_out == 0) return ok();
  // the codes: result element r reads operand index i[d] = dim(operand, d) == 1 ? 0 : r[bdims[d]]
  GatherPlan g;
  std::memset(&g, 0, sizeof g);
  g.in = operand_ptr;
  g.out = result_ptr;
  g.kind = G_PLAIN;
  g.rank = result->rank;
  g.n = n_out;
  int64_t istr[HLO_MAX_RANK];
  strides_of(*operand, istr);
  for (int j = 0; j < result->rank; ++j) {
    const int od = (int)result->minor_to_major[result->rank - 1 - j];
    g.out_size[j] = result->dims[od];
    g.out_logical[j] = od;
  }
  for (int d = 0; d < operand->rank; ++d)
    if (operand->dims[d] != 1) g.in_stride_of_out[broadcast_dimensions[d]] = istr[d];
  for (int k = 0; k < result->rank; ++k) g.perm[k] = k;
  g.in_dt = g.out_dt = S8;
  g.elem_bytes = 1;
  return cuda_status(launch_gather(g, s), "broadcast gather launch");
}

hlo_status hlo_quant_reshape(const hlo_array* operand, const void* operand_ptr, const hlo_quant* operand_q,
                             const hlo_array* result, int32_t result_quantization_dimension, void* result_ptr,
                             void* stream) {
  hlo_status st = check_array(operand, "reshape operand");
  if (st != HLO_OK) return st;
  if ((st = check_array(result, "reshape result")) != HLO_OK) return st;
  if (operand->dtype != result->dtype)
    return fail(HLO_ERR_INVALID_ARG, "reshape (C1): result element type differs from the operand's");
  const int64_t n = numel(*operand);
  if (numel(*result) != n) return fail(HLO_ERR_INVALID_ARG, "reshape (C2): %lld elements into %lld", (long long)n,
                                       (long long)numel(*result));
  if (operand_q) {
    QuantParams qp;
    if (operand->dtype != S8) return fail(HLO_ERR_UNSUPPORTED, "quantized reshape: storage type must be s8");
    if ((st = check_quant(operand_q, *operand, "reshape operand", &qp)) != HLO_OK) return st;
    if (qp.axis < 0) {
      if (result_quantization_dimension != -1)
        return fail(HLO_ERR_INVALID_ARG, "reshape (C1): a per-tensor operand gives a per-tensor result");
    } else {
      const int qd = qp.axis, rqd = result_quantization_dimension;
      if (rqd < 0 || rqd >= result->rank)
        return fail(HLO_ERR_INVALID_ARG, "reshape (C3): result quantization dimension %d out of range", rqd);
      int64_t before_o = 1, after_o = 1, before_r = 1, after_r = 1;
      for (int d = 0; d < qd; ++d) before_o *= operand->dims[d];
      for (int d = qd + 1; d < operand->rank; ++d) after_o *= operand->dims[d];
      for (int d = 0; d < rqd; ++d) before_r *= result->dims[d];
      for (int d = rqd + 1; d < result->rank; ++d) after_r *= result->dims[d];
      if (before_o != before_r || operand->dims[qd] != result->dims[rqd] || after_o != after_r)
        return fail(HLO_ERR_INVALID_ARG, "reshape (C3): result dimension %d does not keep the quantized axis intact", rqd);
    }
  } else if (result_quantization_dimension != -1) {
    return fail(HLO_ERR_INVALID_ARG, "reshape: a quantization dimension without operand parameters");
  }
  const int eb = dt_bytes(operand->dtype);
  if (n > 0 && (!operand_ptr || !result_ptr)) return fail(HLO_ERR_INVALID_ARG, "reshape: NULL data pointer");
  if (ranges_overlap(operand_ptr, n * eb, result_ptr, n * eb))
    return fail(HLO_ERR_INVALID_ARG, "reshape: operand and result overlap");
  if (n == 0) return ok();
  ReshapePlan p;
  std::memset(&p, 0, sizeof p);
  p.in = operand_ptr;
  p.out = result_ptr;
  p.n = n;
  p.elem_bytes = eb;
  int64_t ostr[HLO_MAX_RANK], lex_r[HLO_MAX_RANK];
  strides_of(*operand, ostr);
  int64_t acc = 1;
  for (int d = result->rank - 1; d >= 0; --d) {
    lex_r[d] = acc;
    acc *= result->dims[d];
  }
  std::vector<int64_t> sz, st2;
  for (int k = result->rank - 1; k >= 0; --k) {  // result physical axes, major first
    const int d = (int)result->minor_to_major[k];
    sz.push_back(result->dims[d]);
    st2.push_back(lex_r[d]);
  }
  p.out_to_lex = make_map(sz, st2);
  sz.clear();
  st2.clear();
  for (int d = 0; d < operand->rank; ++d) {  // lexicographic axes of the operand, major first
    sz.push_back(operand->dims[d]);
    st2.push_back(ostr[d]);
  }
  p.lex_to_in = make_map(sz, st2);
  HLO_INJECT("hlo_quant_reshape");
  const cudaStream_t s = as_stream(stream);
  if (p.out_to_lex.identity && p.lex_to_in.identity)
    return cuda_status(launch_copy(operand_ptr, result_ptr, n * eb, s), "copy launch");
  return cuda_status(launch_reshape(p, s), "reshape launch");
}

hlo_status hlo_device_faults(uint32_t* faults, int32_t clear) {
  if (!faults) return fail(HLO_ERR_INVALID_ARG, "device_faults: faults is NULL");
  *faults = 0;
  unsigned int f = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = read_all_faults(&f, clear != 0);
  hlo_status st = cuda_status(e, "device_faults");
  if (st == HLO_OK) *faults = f;
  return st;
}

hlo_status hlo_selftest_bounded_wait(void* stream) {
  return cuda_status(launch_wait_selftest(as_stream(stream)), "bounded-wait self test launch");
}

int32_t hlo_jit_kernels(void) { return jit_chain_kernels(); }

int64_t hlo_jit_source(const hlo_ew_chain* chain, int32_t dtype, char* buf, int64_t buf_len) {
  if (buf_len < 0 || (buf_len > 0 && !buf)) return -1;
  hlo_array arr;
  std::memset(&arr, 0, sizeof arr);
  arr.rank = 1;
  arr.dtype = dtype;
  arr.dims[0] = 1;
  Chain pro;
  if (dtype != HLO_BF16 && dtype != HLO_F16) return -1;
  if (!chain || make_chain(chain, arr, false, "jit source", &pro) != HLO_OK) return -1;
  std::string src;
  if (!jit_chain_source(pro, dtype, &src)) return -1;
  const int64_t len = (int64_t)src.size();
  if (buf && buf_len > len) std::memcpy(buf, src.c_str(), (size_t)len + 1);
  return len;
}

const char* hlo_last_error(void) { return g_err.c_str(); }

const char* hlo_version(void) { return "hlofusion 0.1 (sm_103a)"; }

size_t hlo_reduce_workspace_size(const hlo_array* in, const int64_t* dimensions, int32_t n_dimensions,
                                 int32_t accum_dtype) {
  if (accum_dtype != HLO_F32 || check_array(in, "reduce input") != HLO_OK || !is_float(in->dtype)) return 0;
  if (n_dimensions < 0 || n_dimensions > in->rank || (n_dimensions > 0 && !dimensions)) return 0;
  bool red[HLO_MAX_RANK] = {false};
  for (int i = 0; i < n_dimensions; ++i) {
    const int64_t d = dimensions[i];
    if (d < 0 || d >= in->rank || red[d]) return 0;
    red[d] = true;
  }
  int64_t rows, len;
  if (numel(*in) == 0 || !row_geometry(*in, red, &rows, &len)) return 0;
  return (size_t)row_split_workspace(rows, row_split_factor(rows, len, dt_bytes(in->dtype)));
}

hlo_status hlo_reduce_fusion(const hlo_array* in, const void* in_ptr, const hlo_ew_chain* prologue,
                             const int64_t* dimensions, int32_t n_dimensions, int32_t kind, double init_value,
                             int32_t accum_dtype, const hlo_array* out, void* out_ptr, void* workspace,
                             size_t workspace_bytes, void* stream) {
  hlo_status st = check_array(in, "reduce input");
  if (st != HLO_OK) return st;
  st = check_array(out, "reduce output");
  if (st != HLO_OK) return st;
  if (kind != HLO_RED_ADD && kind != HLO_RED_MAX) return fail(HLO_ERR_INVALID_ARG, "reduce: unknown body %d", kind);
  if (accum_dtype != HLO_F32) return fail(HLO_ERR_UNSUPPORTED, "reduce: only f32 accumulation is implemented");
  if (!is_float(in->dtype)) return fail(HLO_ERR_UNSUPPORTED, "reduce: input element type %d not supported", in->dtype);
  if (!is_float(out->dtype)) return fail(HLO_ERR_UNSUPPORTED, "reduce: output element type %d not supported", out->dtype);
  if (n_dimensions < 0 || n_dimensions > in->rank)
    return fail(HLO_ERR_INVALID_ARG, "reduce (C4): %d dimensions for rank %d", n_dimensions, in->rank);
  if (n_dimensions > 0 && !dimensions) return fail(HLO_ERR_INVALID_ARG, "reduce: dimensions is NULL");
  bool red[HLO_MAX_RANK] = {false};
  for (int i = 0; i < n_dimensions; ++i) {
    const int64_t d = dimensions[i];
    if (d < 0 || d >= in->rank)
      return fail(HLO_ERR_INVALID_ARG, "reduce (C4): dimension %lld outside [0, %d)", (long long)d, in->rank);
    if (red[d]) return fail(HLO_ERR_INVALID_ARG, "reduce (C5): dimension %lld repeated", (long long)d);
    red[d] = true;
  }
  std::vector<int> kept;
  for (int d = 0; d < in->rank; ++d)
    if (!red[d]) kept.push_back(d);
  if (out->rank != (int)kept.size())
    return fail(HLO_ERR_INVALID_ARG, "reduce (C7): output rank %d, expected %d", out->rank, (int)kept.size());
  for (size_t k = 0; k < kept.size(); ++k)
    if (out->dims[k] != in->dims[kept[k]])
      return fail(HLO_ERR_INVALID_ARG, "reduce (C7): output dim %d is %lld, expected %lld", (int)k,
                  (long long)out->dims[k], (long long)in->dims[kept[k]]);
  Chain chain;
  st = make_chain(prologue, *in, true, "reduce prologue", &chain);
  if (st != HLO_OK) return st;
  const int64_t n_in = numel(*in), n_out = numel(*out);
  if (n_in > 0 && !in_ptr) return fail(HLO_ERR_INVALID_ARG, "reduce: input pointer is NULL");
  if (n_out > 0 && !out_ptr) return fail(HLO_ERR_INVALID_ARG, "reduce: output pointer is NULL");
  if (ranges_overlap(in_ptr, n_in * dt_bytes(in->dtype), out_ptr, n_out * dt_bytes(out->dtype)))
    return fail(HLO_ERR_INVALID_ARG, "reduce: input and output overlap");
  HLO_INJECT("hlo_reduce_fusion");
  const cudaStream_t s = as_stream(stream);
  // init_values has the inputs' element type ("reduce" C2): the literal is rounded to it
  const float init = constant_of_type(init_value, in->dtype);
  if (n_out == 0) return ok();
  int64_t n_red = 1;
  for (int d = 0; d < in->rank; ++d)
    if (red[d]) n_red *= in->dims[d];
  if (n_red == 0) return cuda_status(launch_fill(out_ptr, out->dtype, n_out, init, s), "fill kernel launch");

  int64_t istr[HLO_MAX_RANK], ostr_out[HLO_MAX_RANK];
  strides_of(*in, istr);
  strides_of(*out, ostr_out);
  int64_t ostr_in[HLO_MAX_RANK] = {0};  // output stride of each kept INPUT logical dim
  for (size_t k = 0; k < kept.size(); ++k) ostr_in[kept[k]] = ostr_out[k];

  // physical axes of the input, major first, unit dims dropped; runs of reduced / kept dims
  struct Run {
    bool reduced;
    int64_t size;
    std::vector<int> dims;
  };
  std::vector<Run> runs;
  for (int k = in->rank - 1; k >= 0; --k) {
    const int d = (int)in->minor_to_major[k];
    if (in->dims[d] == 1) continue;
    if (!runs.empty() && runs.back().reduced == red[d]) {
      runs.back().size *= in->dims[d];
      runs.back().dims.push_back(d);
    } else {
      runs.push_back({red[d], in->dims[d], {d}});
    }
  }
  int n_red_runs = 0;
  for (auto& r : runs) n_red_runs += r.reduced ? 1 : 0;
  // kept dims in input physical order (major first), for the row -> output / broadcast maps
  std::vector<int> kept_phys;
  for (auto& r : runs)
    if (!r.reduced)
      for (int d : r.dims) kept_phys.push_back(d);
  auto kept_map = [&](const int64_t* target_stride_by_dim) {
    std::vector<int64_t> sz, st2;
    for (int d : kept_phys) {
      sz.push_back(in->dims[d]);
      st2.push_back(target_stride_by_dim[d]);
    }
    return make_map(sz, st2);
  };

  const bool has_bcast = chain_has_bcast(chain);
  const bool row_pattern = n_red_runs == 0 || (n_red_runs == 1 && runs.back().reduced);
  const bool col_pattern = n_red_runs == 1 && !runs.back().reduced;

  if (row_pattern) {
    RowReducePlan p;
    std::memset(&p, 0, sizeof p);
    p.in = in_ptr;
    p.out = out_ptr;
    p.len = n_red_runs ? runs.back().size : 1;
    p.rows = n_in / p.len;
    p.in_dt = in->dtype;
    p.out_dt = out->dtype;
    p.kind = kind;
    p.init = init;
    p.chain = chain;
    p.omap = kept_map(ostr_in);
    p.bmode = BC_NONE;
    p.split = 1;
    p.seg = p.len;
    // few long rows: split them into segments reduced by separate blocks (partials in the workspace)
    const int64_t split = row_split_factor(p.rows, p.len, dt_bytes(in->dtype));
    if (split > 1) {
      int64_t seg = (p.len + split - 1) / split;
      seg = (seg + 511) / 512 * 512;  // whole 16-byte vectors in every segment
      const int64_t nsplit = (p.len + seg - 1) / seg;
      const int64_t need = row_split_workspace(p.rows, nsplit);
      if (workspace && (int64_t)workspace_bytes < need)
        return fail(HLO_ERR_WORKSPACE, "reduce: workspace of %zu bytes, %lld needed (hlo_reduce_workspace_size)",
                    workspace_bytes, (long long)need);
      if (workspace && nsplit > 1) {
        if ((uintptr_t)workspace % 4 != 0) return fail(HLO_ERR_INVALID_ARG, "reduce: workspace is not 4-byte aligned");
        if (ranges_overlap(workspace, need, in_ptr, n_in * dt_bytes(in->dtype)) ||
            ranges_overlap(workspace, need, out_ptr, n_out * dt_bytes(out->dtype)))
          return fail(HLO_ERR_INVALID_ARG, "reduce: workspace overlaps the input or the output");
        p.split = nsplit;
        p.seg = seg;
        p.ws = static_cast<float*>(workspace);
      }
    }
    bool ok_plan = true;
    if (has_bcast) {
      bool kept_zero = true, red_match = true, red_zero = true;
      for (int d = 0; d < in->rank; ++d) {
        if (in->dims[d] == 1) continue;
        if (red[d]) {
          if (chain.bstride[d] != istr[d]) red_match = false;
          if (chain.bstride[d] != 0) red_zero = false;
        } else if (chain.bstride[d] != 0) {
          kept_zero = false;
        }
      }
      if (kept_zero && red_match && n_red_runs == 1) {
        p.bmode = BC_ROWVEC;
      } else if (red_zero) {
        p.bmode = BC_PERROW;
        p.bmap = kept_map(chain.bstride);
      } else {
        ok_plan = false;
      }
    }
    if (ok_plan) return cuda_status(launch_row_reduce(p, s), "row reduce launch");
  } else if (col_pattern && !has_bcast) {
    ColReducePlan p;
    std::memset(&p, 0, sizeof p);
    p.in = in_ptr;
    p.out = out_ptr;
    p.a = 1;
    p.b = 1;
    bool before = true;
    for (auto& r : runs) {
      if (r.reduced) {
        p.r = r.size;
        before = false;
      } else if (before) {
        p.a *= r.size;
      } else {
        p.b *= r.size;
      }
    }
    p.in_dt = in->dtype;
    p.out_dt = out->dtype;
    p.kind = kind;
    p.init = init;
    p.chain = chain;
    p.omap = kept_map(ostr_in);
    if (p.a <= 65535) return cuda_status(launch_col_reduce(p, s), "column reduce launch");
  }

  // general plan
  GenReducePlan g;
  std::memset(&g, 0, sizeof g);
  g.in = in_ptr;
  g.out = out_ptr;
  g.in_dt = in->dtype;
  g.out_dt = out->dtype;
  g.kind = kind;
  g.init = init;
  g.chain = chain;
  g.n_out = n_out;
  g.n_red = n_red;
  g.rank = in->rank;
  g.nk = out->rank;
  for (int j = 0; j < out->rank; ++j) {
    const int od = (int)out->minor_to_major[out->rank - 1 - j];
    g.kdim_size[j] = out->dims[od];
    g.kdim_logical[j] = kept[od];
    g.kdim_in_stride[j] = istr[kept[od]];
  }
  for (int k = in->rank - 1; k >= 0; --k) {
    const int d = (int)in->minor_to_major[k];
    if (!red[d]) continue;
    g.rdim_size[g.nr] = in->dims[d];
    g.rdim_in_stride[g.nr] = istr[d];
    g.rdim_logical[g.nr] = d;
    ++g.nr;
  }
  return cuda_status(launch_gen_reduce(g, s), "general reduce launch");
}

hlo_status hlo_transpose_fusion(const hlo_array* in, const void* in_ptr, const hlo_ew_chain* prologue,
                                const int64_t* permutation, int32_t self_add_epilogue, const hlo_ew_chain* epilogue,
                                const hlo_array* out, void* out_ptr, void* stream) {
  hlo_status st = check_array(in, "transpose input");
  if (st != HLO_OK) return st;
  st = check_array(out, "transpose output");
  if (st != HLO_OK) return st;
  if (out->rank != in->rank) return fail(HLO_ERR_INVALID_ARG, "transpose: output rank differs from input rank");
  if (out->dtype != in->dtype) return fail(HLO_ERR_INVALID_ARG, "transpose: output element type differs from input");
  if (in->rank > 0 && !permutation) return fail(HLO_ERR_INVALID_ARG, "transpose: permutation is NULL");
  bool seen[HLO_MAX_RANK] = {false};
  for (int k = 0; k < in->rank; ++k) {
    const int64_t p = permutation[k];
    if (p < 0 || p >= in->rank || seen[p])
      return fail(HLO_ERR_INVALID_ARG, "transpose: permutation is not a permutation of 0..%d", in->rank - 1);
    seen[p] = true;
    if (out->dims[k] != in->dims[p])
      return fail(HLO_ERR_INVALID_ARG, "transpose: output dim %d is %lld, expected dims(in)[%lld] = %lld", k,
                  (long long)out->dims[k], (long long)p, (long long)in->dims[p]);
    if (self_add_epilogue && out->dims[k] != in->dims[k])
      return fail(HLO_ERR_INVALID_ARG, "transpose: the self-add form needs dims(out) == dims(in) (add C1)");
  }
  Chain pro, epi;
  st = make_chain(prologue, *in, true, "transpose prologue", &pro);
  if (st != HLO_OK) return st;
  st = make_chain(epilogue, *out, false, "transpose epilogue", &epi);
  if (st != HLO_OK) return st;
  const int64_t n = numel(*in);
  const int64_t bytes = n * dt_bytes(in->dtype);
  if (n > 0 && (!in_ptr || !out_ptr)) return fail(HLO_ERR_INVALID_ARG, "transpose: NULL data pointer");
  if (ranges_overlap(in_ptr, bytes, out_ptr, bytes)) return fail(HLO_ERR_INVALID_ARG, "transpose: input and output overlap");
  if (n == 0) return ok();
  HLO_INJECT("hlo_transpose_fusion");
  const cudaStream_t s = as_stream(stream);
  const bool bcast = chain_has_bcast(pro);

  if (self_add_epilogue) {
    // fast pair-tile path: a square matrix once unit dims are dropped, transposed, same memory order
    std::vector<int> nonunit;
    for (int d = 0; d < in->rank; ++d)
      if (in->dims[d] != 1) nonunit.push_back(d);
    bool pair = in->dtype == F32 && !bcast && nonunit.size() == 2;
    if (pair) {
      const int da = nonunit[0], db = nonunit[1];
      pair = in->dims[da] == in->dims[db] && permutation[da] == db && permutation[db] == da;
      auto minor_of = [&](const hlo_array& a) {
        for (int k = 0; k < a.rank; ++k)
          if (a.dims[a.minor_to_major[k]] != 1) return (int)a.minor_to_major[k];
        return -1;
      };
      pair = pair && minor_of(*in) == minor_of(*out);
    }
    // the pair kernels index tile pairs with 31-bit counts: n < 64 * 65536 (far beyond any device's memory)
    if (pair && in->dims[nonunit[0]] >= (int64_t)64 * 65536) pair = false;
    if (pair) {
      SelfAddPlan p;
      std::memset(&p, 0, sizeof p);
      p.in = in_ptr;
      p.out = out_ptr;
      p.n = in->dims[nonunit[0]];
      p.dt = in->dtype;
      p.pro = pro;
      p.epi = epi;
      return cuda_status(launch_selfadd_transpose(p, s), "self-add transpose launch");
    }
    return plan_gather_plain(*in, in_ptr, *out, out_ptr, permutation, 1, pro, epi, s);
  }
  if (bcast) return plan_gather_plain(*in, in_ptr, *out, out_ptr, permutation, 0, pro, epi, s);

  Canon c = canonicalize(*in, permutation, out->minor_to_major);
  bool identity = true;
  for (int j = 0; j < c.k; ++j)
    if (c.out_pos[j] != j) identity = false;
  if (identity) {
    if (pro.n == 0 && epi.n == 0) return cuda_status(launch_copy(in_ptr, out_ptr, bytes, s), "copy launch");
    return cuda_status(launch_elementwise(in_ptr, out_ptr, n, in->dtype, pro, epi, s), "elementwise launch");
  }
  const int ax_a = c.k - 1;
  int ax_b = -1;
  for (int j = 0; j < c.k; ++j)
    if (c.out_pos[j] == c.k - 1) ax_b = j;
  if (ax_b == ax_a || ax_b < 0) return plan_gather_plain(*in, in_ptr, *out, out_ptr, permutation, 0, pro, epi, s);
  TilePlan t;
  std::memset(&t, 0, sizeof t);
  t.in = in_ptr;
  t.out = out_ptr;
  t.k = c.k;
  int64_t sacc = 1;
  for (int j = c.k - 1; j >= 0; --j) {
    t.size[j] = c.size[j];
    t.in_stride[j] = sacc;
    sacc *= c.size[j];
  }
  // output strides: axes ordered by out_pos, minor (largest position) first
  std::vector<int> by_pos(c.k);
  for (int j = 0; j < c.k; ++j) by_pos[c.out_pos[j]] = j;
  sacc = 1;
  for (int q = c.k - 1; q >= 0; --q) {
    t.out_stride[by_pos[q]] = sacc;
    sacc *= c.size[by_pos[q]];
  }
  t.ax_a = ax_a;
  t.ax_b = ax_b;
  t.n_batch = 1;
  for (int j = 0; j < c.k; ++j) {
    if (j == ax_a || j == ax_b) continue;
    t.batch_axis[t.nbatch_axes++] = j;
    t.n_batch *= c.size[j];
  }
  t.dt = in->dtype;
  t.pro = pro;
  t.epi = epi;
  return cuda_status(launch_tile_transpose(t, s), "tiled transpose launch");
}

hlo_status hlo_layout_convert(const hlo_array* in, const void* in_ptr, const int64_t* out_minor_to_major,
                              void* out_ptr, void* stream) {
  hlo_status st = check_array(in, "layout_convert input");
  if (st != HLO_OK) return st;
  if (in->rank > 0 && !out_minor_to_major) return fail(HLO_ERR_INVALID_ARG, "layout_convert: out_minor_to_major is NULL");
  hlo_array out = *in;
  for (int k = 0; k < in->rank; ++k) out.minor_to_major[k] = out_minor_to_major[k];
  st = check_array(&out, "layout_convert output");
  if (st != HLO_OK) return st;
  int64_t perm[HLO_MAX_RANK];
  for (int k = 0; k < in->rank; ++k) perm[k] = k;
  HLO_INJECT("hlo_layout_convert");
  return hlo_transpose_fusion(in, in_ptr, nullptr, perm, 0, nullptr, &out, out_ptr, stream);
}

hlo_status hlo_quant_fusion(const hlo_array* in, const void* in_ptr, const hlo_quant* in_q,
                            const hlo_ew_chain* float_ops, const int64_t* out_minor_to_major, const hlo_array* out,
                            void* out_ptr, const hlo_quant* out_q, void* stream) {
  hlo_status st = check_array(in, "quant input");
  if (st != HLO_OK) return st;
  st = check_array(out, "quant output");
  if (st != HLO_OK) return st;
  if (in->dtype != S8) return fail(HLO_ERR_UNSUPPORTED, "quant: storage type must be s8");
  if (out->rank != in->rank) return fail(HLO_ERR_INVALID_ARG, "quant: output rank differs from input rank");
  for (int d = 0; d < in->rank; ++d)
    if (out->dims[d] != in->dims[d]) return fail(HLO_ERR_INVALID_ARG, "quant: a layout change keeps the shape; dim %d differs", d);
  if (in->rank > 0 && out_minor_to_major)
    for (int k = 0; k < in->rank; ++k)
      if (out->minor_to_major[k] != out_minor_to_major[k])
        return fail(HLO_ERR_INVALID_ARG, "quant: out_minor_to_major differs from out->minor_to_major");
  QuantParams qin, qout;
  std::memset(&qout, 0, sizeof qout);
  st = check_quant(in_q, *in, "quant input parameters", &qin);
  if (st != HLO_OK) return st;
  const bool out_float = out_q == nullptr;
  if (out_float) {
    if (out->dtype != F32) return fail(HLO_ERR_INVALID_ARG, "quant: without output parameters the output must be f32");
  } else {
    if (out->dtype != S8) return fail(HLO_ERR_UNSUPPORTED, "quant: quantized output storage must be s8");
    st = check_quant(out_q, *out, "quant output parameters", &qout);
    if (st != HLO_OK) return st;
  }
  Chain ops;
  st = make_chain(float_ops, *in, true, "quant float ops", &ops, F32);
  if (st != HLO_OK) return st;
  const int64_t n = numel(*in);
  if (n > 0 && (!in_ptr || !out_ptr)) return fail(HLO_ERR_INVALID_ARG, "quant: NULL data pointer");
  if (ranges_overlap(in_ptr, n, out_ptr, n * dt_bytes(out->dtype)))
    return fail(HLO_ERR_INVALID_ARG, "quant: input and output overlap");
  if (n == 0) return ok();
  HLO_INJECT("hlo_quant_fusion");
  const cudaStream_t s = as_stream(stream);

  // fast path: two non-unit dims (i major, j minor in the input), output with i minor
  std::vector<int> nonunit;
  for (int d = 0; d < in->rank; ++d)
    if (in->dims[d] != 1) nonunit.push_back(d);
  auto minor_of = [&](const hlo_array& a) {
    for (int k = 0; k < a.rank; ++k)
      if (a.dims[a.minor_to_major[k]] != 1) return (int)a.minor_to_major[k];
    return -1;
  };
  if (!out_float && nonunit.size() == 2 && !chain_has_bcast(ops)) {
    const int jd = minor_of(*in);
    const int id = nonunit[0] == jd ? nonunit[1] : nonunit[0];
    if (minor_of(*out) == id) {
      auto axis_of = [&](int qd) { return qd < 0 ? -1 : qd == id ? 0 : qd == jd ? 1 : -2; };
      const int ain = axis_of(qin.axis), aout = axis_of(qout.axis);
      if (ain != -2 && aout != -2) {
        QuantTilePlan p;
        std::memset(&p, 0, sizeof p);
        p.in = reinterpret_cast<const int8_t*>(in_ptr);
        p.out = reinterpret_cast<int8_t*>(out_ptr);
        p.n0 = in->dims[id];
        p.n1 = in->dims[jd];
        p.qin = qin;
        p.qin.axis = ain;
        p.qout = qout;
        p.qout.axis = aout;
        p.ops = ops;
        return cuda_status(launch_quant_tile(p, s), "quantized tile launch");
      }
    }
  }
  GatherPlan g;
  std::memset(&g, 0, sizeof g);
  g.in = in_ptr;
  g.out = out_ptr;
  g.kind = G_QUANT;
  g.rank = in->rank;
  g.n = n;
  int64_t istr[HLO_MAX_RANK];
  strides_of(*in, istr);
  for (int j = 0; j < out->rank; ++j) {
    const int od = (int)out->minor_to_major[out->rank - 1 - j];
    g.out_size[j] = out->dims[od];
    g.out_logical[j] = od;
  }
  for (int k = 0; k < in->rank; ++k) {
    g.perm[k] = k;
    g.in_stride_of_out[k] = istr[k];
  }
  g.in_dt = S8;
  g.out_dt = out->dtype;
  g.elem_bytes = 1;
  g.pro = ops;
  g.qin = qin;
  g.qout = qout;
  g.qin_axis_out = qin.axis;
  g.qout_axis_out = out_float ? -1 : qout.axis;
  g.out_float = out_float ? 1 : 0;
  return cuda_status(launch_gather(g, s), "quantized gather launch");
}

}  // extern "C"

// ---- reduce without a caller workspace ------------------------------------------------------------------
// hlo_reduce_fusion needs a device workspace for row reductions it splits across blocks (few long rows).
// A caller that cannot allocate device memory where it runs the reduce -- code embedded in another
// runtime that owns all device memory through its own allocator, or running under a memory budget fixed
// when it started -- has none to give. For those callers the library keeps one fixed scratch array per
// device, in this file, and hlo_reduce_fusion_noalloc passes it as the workspace.
namespace {
constexpr size_t kNoAllocScratchBytes = 64 * 1024;  // room for 16384 f32 row-segment partials
}  // namespace

// The scratch itself: every device that loads the library holds it until the process exits. In host
// code its name is only a host-side stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress below, once per device, and that address is what the kernels receive.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

// Device address of the scratch on the current device, looked up on the first call per device.
static hlo_status noalloc_scratch(void** ptr) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e, "reduce_fusion_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= 64)
    return fail(HLO_ERR_UNSUPPORTED, "reduce_fusion_noalloc: device %d beyond the 64 this library tracks", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_status(e, "reduce_fusion_noalloc: cudaGetSymbolAddress of the scratch");
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return HLO_OK;
}

extern "C" hlo_status hlo_reduce_fusion_noalloc(const hlo_array* in, const void* in_ptr, const hlo_ew_chain* prologue,
                                                const int64_t* dimensions, int32_t n_dimensions, int32_t kind,
                                                double init_value, int32_t accum_dtype, const hlo_array* out,
                                                void* out_ptr, void* stream) {
  const size_t need = hlo_reduce_workspace_size(in, dimensions, n_dimensions, accum_dtype);
  if (need > kNoAllocScratchBytes)
    return fail(HLO_ERR_WORKSPACE,
                "reduce_fusion_noalloc: this reduction needs %zu bytes of scratch, more than the %zu the library "
                "keeps per device; use hlo_reduce_fusion with a workspace",
                need, kNoAllocScratchBytes);
  HLO_INJECT("hlo_reduce_fusion_noalloc");
  void* scratch = nullptr;
  if (need > 0) {
    const hlo_status st = noalloc_scratch(&scratch);
    if (st != HLO_OK) return st;
  }
  return hlo_reduce_fusion(in, in_ptr, prologue, dimensions, n_dimensions, kind, init_value, accum_dtype, out, out_ptr,
                           scratch, scratch ? kNoAllocScratchBytes : 0, stream);
}
