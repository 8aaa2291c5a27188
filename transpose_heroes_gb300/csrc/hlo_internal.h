// Internal plan structures shared by the host planner (hlo_api.cu) and the kernel translation units.
// Every structure here is plain data passed to kernels by value.
#pragma once
#include <cstddef>
#include <cstdint>
#include <string>

#include <cuda_runtime.h>

namespace hlo {

enum Dt : int { F32 = 0, BF16 = 1, S8 = 2, F16 = 3, S32 = 4 };
enum Op : int {
  OP_NONE = 0, OP_EXP = 1, OP_LOG = 2, OP_ABS = 3, OP_NEG = 4, OP_ADD_BCAST = 5, OP_TANH = 6,
  OP_ADD_CONST = 7, OP_MUL_CONST = 8, OP_ADD_IN = 9, OP_MUL_IN = 10
};
enum Red : int { RED_ADD = 0, RED_MAX = 1 };

constexpr int kMaxRank = 8;
constexpr int kMaxOps = 16;

inline __host__ __device__ int dt_bytes(int dt) {
  return dt == F32 || dt == S32 ? 4 : dt == BF16 || dt == F16 ? 2 : dt == S8 ? 1 : 0;
}

// A linear index decomposed over up to kMaxRank axes (major first) and re-composed with other
// strides: offset(k) = sum_j ((k / inner_j) % size_j) * stride_j. Used for "row k -> output offset"
// and "row k -> broadcast offset" maps. identity != 0 means offset(k) == k.
struct IndexMap {
  int n;
  int identity;
  int64_t size[kMaxRank];
  int64_t stride[kMaxRank];
};

__host__ __device__ inline int64_t map_index(const IndexMap& m, int64_t k) {
  if (m.identity) return k;
  int64_t off = 0;
  for (int j = m.n - 1; j >= 0; --j) {
    int64_t s = m.size[j];
    off += (k % s) * m.stride[j];
    k /= s;
  }
  return off;
}

// Elementwise chain as the kernels see it. dt is the element type of the array the chain is
// attached to; round16 = round every op result to dt (16-bit float types only).
// Broadcast operand: bptr/bdt and, for the general kernels, bstride[d] = offset contribution of the
// fused array's logical index in dimension d (0 where the operand is broadcast).
struct Chain {
  int n;
  int op[kMaxOps];
  float imm[kMaxOps];  // constants of OP_ADD_CONST / OP_MUL_CONST, already values of the element type
  int round16;
  int dt;
  const void* bptr;
  int bdt;
  int64_t bstride[kMaxRank];
};

// Broadcast addressing in the fast row-reduce kernel.
enum BcastMode : int { BC_NONE = 0, BC_ROWVEC = 1, BC_PERROW = 2 };

struct RowReducePlan {
  const void* in;
  void* out;
  int64_t rows;     // K
  int64_t len;      // R, elements per row (contiguous)
  int in_dt, out_dt, kind;
  float init;
  Chain chain;
  int bmode;        // BcastMode
  IndexMap bmap;    // BC_PERROW: row -> broadcast offset
  IndexMap omap;    // row -> output offset
  // split rows: with split > 1 every row is cut into `split` segments of `seg` elements (the last one
  // shorter); the blocks reduce segments into ws[row * split + segment], and a second kernel combines
  // each row's partials in segment order
  int64_t split;
  int64_t seg;
  float* ws;
};

// Segments per row for a row reduce of `rows` rows of `len` elements of `eb` bytes on this device:
// 1 (no split) unless the rows are too few to occupy the device and long enough to share out.
int64_t row_split_factor(int64_t rows, int64_t len, int eb);
// Workspace bytes a split row reduce needs (0 without a split).
inline int64_t row_split_workspace(int64_t rows, int64_t split) { return split > 1 ? rows * split * 4 : 0; }

struct ColReducePlan {
  const void* in;
  void* out;
  int64_t a, r, b;  // [A, R, B] in physical order, B contiguous
  int in_dt, out_dt, kind;
  float init;
  Chain chain;      // no broadcast in this kernel
  IndexMap omap;    // (a * B + b) -> output offset
};

// General reduce: one thread per output element.
struct GenReducePlan {
  const void* in;
  void* out;
  int in_dt, out_dt, kind;
  float init;
  Chain chain;
  int64_t n_out, n_red;
  // output element (linear index in output physical order) -> logical kept index
  int nk;
  int64_t kdim_size[kMaxRank];     // kept axes in output physical order (major first)
  int64_t kdim_in_stride[kMaxRank];
  int kdim_logical[kMaxRank];      // logical dimension of the input
  int nr;
  int64_t rdim_size[kMaxRank];     // reduced axes in input physical order (major first)
  int64_t rdim_in_stride[kMaxRank];
  int rdim_logical[kMaxRank];
  int rank;
};

// Pair-tile transpose with self add: out = f(in) + f(in)^T for a square 2-D array (after removing
// unit dimensions) with identical input/output layouts; physically [n, n] row-major.
struct SelfAddPlan {
  const void* in;
  void* out;
  int64_t n;
  int dt;
  Chain pro, epi;
};

// Tiled transpose of canonical physical axes: input axes 0..k-1 (major..minor, contiguous strides),
// output written with out_stride per axis. Axis a_in = k-1 (input-minor), axis b = output-minor.
struct TilePlan {
  const void* in;
  void* out;
  int k;
  int64_t size[kMaxRank];
  int64_t in_stride[kMaxRank];
  int64_t out_stride[kMaxRank];
  int ax_a;           // input-minor axis (stride 1 in input)
  int ax_b;           // output-minor axis (stride 1 in output)
  int64_t n_batch;    // product of the other axes
  int nbatch_axes;
  int batch_axis[kMaxRank];
  int dt;             // element type
  Chain pro, epi;     // f32 chains only (no broadcast)
};

// Quantized relayout of a 2-D s8 array: logical [n0, n1], input row-major (dim 1 minor), output
// column-major (dim 0 minor); per-axis or per-tensor dequantize, quantize per-tensor or per-axis.
struct QuantParams {
  int axis;                 // quantization dimension in the 2-D canonical view: 0, 1 or -1
  const float* scales;      // device, when per-axis
  const int32_t* zps;       // device, when per-axis
  float scale;              // per-tensor
  int32_t zp;               // per-tensor
  float inv_scale;          // per-tensor: RN(1 / scale), used by the division shortcut
  int32_t smin, smax;
  float max_abs_scale;      // largest |scale| when the host copy was given, else -1 (unknown)
};

struct QuantTilePlan {
  const int8_t* in;
  int8_t* out;
  int64_t n0, n1;
  QuantParams qin, qout;
  Chain ops;                // f32 chain on the dequantized value (no broadcast)
};

// General elementwise gather: one thread per output element (output physical order).
// Covers transposes, layout changes and quantized relayouts the fast kernels do not.
enum GatherKind : int { G_PLAIN = 0, G_QUANT = 1 };
struct GatherPlan {
  const void* in;
  void* out;
  int kind;
  int rank;
  int64_t n;
  int64_t out_size[kMaxRank];       // output logical dims in output physical order (major first)
  int out_logical[kMaxRank];        // output logical dimension of each physical axis
  int64_t in_stride_of_out[kMaxRank];   // input stride for each output logical dim (via permutation)
  int64_t self_stride_of_out[kMaxRank]; // self-add: input stride of the same logical index
  int self_add;
  int in_dt, out_dt;
  int elem_bytes;
  Chain pro, epi;                   // pro.bstride is per INPUT logical dim, epi has no broadcast
  int perm[kMaxRank];               // out logical dim k reads input logical dim perm[k]
  // quant
  int qin_axis_out;                 // output logical dim of the input quantization axis (-1)
  int qout_axis_out;                // output logical dim of the output quantization axis (-1)
  QuantParams qin, qout;
  int out_float;                    // quant with float output
};

// Kernel launchers (defined in the k_*.cu translation units). Return the launch status.
// Max/argmax variadic reduce. Output o (lexicographic over the kept dims): V at
// map_index(vkept, o) + map_index(vred, t) for walk position t; K (if any) likewise with kkept/kred;
// results at map_index(okept, o) and map_index(ikept, o).
struct ArgmaxPlan {
  const void* v;
  const int32_t* k;  // NULL: the index is the walk position
  void* out;
  int32_t* out_idx;
  int dt;
  int64_t n_out, n_red;
  IndexMap vkept, vred, kkept, kred, okept, ikept;
  float init_value;
  int32_t init_index;
};
cudaError_t launch_argmax(const ArgmaxPlan& p, cudaStream_t s);

// Quantized binary op: out at map_index(omap, i) = q(op(dq(lhs at lmap(i)), dq(rhs at rmap(i)))), i the
// logical linear index (identity maps when all three share one layout).
struct QuantBinaryPlan {
  const int8_t* lhs;
  const int8_t* rhs;
  int8_t* out;
  int64_t n;
  int op;
  IndexMap lmap, rmap, omap;
  QuantParams ql, qr, qo;
};
cudaError_t launch_quant_binary(const QuantBinaryPlan& p, cudaStream_t s);

// Reshape: output element e (physical order) is the element at lexicographic position
// p = map_index(out_to_lex, e) of the operand, found at map_index(lex_to_in, p).
struct ReshapePlan {
  const void* in;
  void* out;
  int64_t n;
  int elem_bytes;
  IndexMap out_to_lex, lex_to_in;
};
cudaError_t launch_reshape(const ReshapePlan& p, cudaStream_t s);
// Quantization parameters of a result: n pairs, each copied from (src_s, src_z)[single ? 0 : i], or, with
// src_s == NULL, the pair (s0, z0) repeated.
cudaError_t launch_quant_params(const float* src_s, const int32_t* src_z, float s0, int32_t z0, int single, float* dst_s,
                                int32_t* dst_z, int64_t n, cudaStream_t s);
// Device-side faults (bit mask, the same values as HLO_FAULT_* of the C ABI).
constexpr unsigned int kFaultCopyTimeout = 1u;
// Every translation unit whose kernels record faults has its own device fault word; it registers a
// reader of that word (copy out, clear when asked; the caller has waited for the device) when the
// library is loaded. read_all_faults ORs the words of every registered unit.
using FaultReader = cudaError_t (*)(unsigned int* faults, bool clear);
int register_fault_reader(FaultReader r);
cudaError_t read_all_faults(unsigned int* faults, bool clear);
// Launches the bounded-wait self test (sets kFaultCopyTimeout after about a millisecond).
cudaError_t launch_wait_selftest(cudaStream_t s);
cudaError_t launch_row_reduce(const RowReducePlan& p, cudaStream_t s);
cudaError_t launch_col_reduce(const ColReducePlan& p, cudaStream_t s);
cudaError_t launch_gen_reduce(const GenReducePlan& p, cudaStream_t s);
cudaError_t launch_fill(void* out, int dt, int64_t n, float value, cudaStream_t s);
cudaError_t launch_selfadd_transpose(const SelfAddPlan& p, cudaStream_t s);
cudaError_t launch_tile_transpose(const TilePlan& p, cudaStream_t s);
cudaError_t launch_quant_tile(const QuantTilePlan& p, cudaStream_t s);
cudaError_t launch_gather(const GatherPlan& p, cudaStream_t s);
cudaError_t launch_copy(const void* in, void* out, int64_t nbytes, cudaStream_t s);
cudaError_t launch_elementwise(const void* in, void* out, int64_t n, int dt, const Chain& pro, const Chain& epi,
                               cudaStream_t s);

// Run-time generated 16-bit chain kernels (jit_chain.cu): whether the generator writes this chain;
// the launch (`used` false when no kernel could be built: the caller runs the interpreter); the number
// of kernels built for the current device (-1 when NVRTC or the driver calls are unavailable).
bool jit_chain_ok(const Chain& pro, const Chain& epi, int dt);
cudaError_t launch_jit_chain(const void* in, void* out, int64_t n, int dt, const Chain& pro, cudaStream_t s, bool* used);
int jit_chain_kernels();
// The CUDA source generated for a chain the generator takes (with a run-table slot free); false for
// any other chain. No device work.
bool jit_chain_source(const Chain& pro, int dt, std::string* out);
// Device address of the bf16 tanh table (k_elementwise.cu), or NULL.
const void* tanh_table_address();

// Device properties cached per device (SM count, cluster support).
int device_sm_count();

// Resident blocks per SM of `kernel` at this block size and dynamic shared memory, cached per kernel
// and device; on first use also raises the kernel's dynamic shared-memory limit to `smem`.
int kernel_blocks_per_sm(const void* kernel, int threads, size_t smem);
// Cluster size (the largest of 8, 4, 2 that fits) and the number of clusters that can be resident at
// once, for a kernel with one block per SM; sets the kernel's dynamic shared-memory limit. Cached.
// (On GB300, 15 clusters of 8 fit: 120 SMs. Smaller clusters reach more SMs but each block then
// builds a larger share of its table, which measured slower for the 16-bit chain tables.)
void table_cluster_shape(const void* kernel, int threads, size_t smem, int* cluster_size, int* clusters);

}  // namespace hlo
