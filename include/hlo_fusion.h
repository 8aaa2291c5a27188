/*
 * hlo_fusion.h -- C ABI of libhlofusion: HLO fusions whose hero is a reduce, a transpose or a layout
 * change, executed on one GB300 GPU (sm_103a) by hand-written CUDA kernels.
 *
 * Every fusion reads its inputs from HBM once and writes its output once; the elementwise prologue
 * and epilogue (exp, log, abs, negate, add of a broadcast operand) and uniform (de)quantization are
 * applied in registers.
 *
 * Conventions shared by all entry points
 * --------------------------------------
 *  - Arrays are described by hlo_array: a logical shape (dims, numbered 0..rank-1, each >= 0; size 0
 *    is valid) and a physical layout minor_to_major, a permutation of 0..rank-1 whose first entry is
 *    the minor-most dimension (the one that changes fastest in linear memory). Source: "XLA Shapes and
 *    Layout", sections "Shapes" and "Layout" (minor-to-major ordering, the [2 x 3] example), and
 *    "Default minor-to-major ordering" ([rank-1, ..., 0], i.e. row-major).
 *  - Data pointers (in_ptr, out_ptr, hlo_ew_chain.bcast_ptr, hlo_quant.scales/zero_points) are
 *    DEVICE pointers to dense buffers in that layout. Descriptors are host memory, read during the
 *    call only. The caller owns every buffer; the library allocates no device memory and keeps no
 *    pointer after the call returns.
 *  - stream is a cudaStream_t (NULL = the legacy default stream). Calls are asynchronous: they
 *    validate, enqueue one or more kernels on the stream and return. The output is defined once the
 *    stream reaches that point.
 *  - Inputs and outputs must not overlap (HLO_ERR_INVALID_ARG). Alignment is not required: buffers
 *    that are not 16-byte aligned, or rows whose byte length is not a multiple of 16, take a
 *    narrower-access variant of the same kernel.
 *  - On any error nothing is enqueued, except HLO_ERR_CUDA, which reports a failed launch.
 *    hlo_last_error() returns a thread-local message naming the violated constraint.
 *  - Floating point: reductions accumulate in f32; the order of accumulation is implementation
 *    defined, as the reduce semantics allow ("StableHLO Specification", section "reduce"). exp, log
 *    and tanh are correctly rounded; transposes, layout changes, elementwise chains and quantization
 *    are bit-exact.
 */
#ifndef HLO_FUSION_H
#define HLO_FUSION_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HLO_MAX_RANK 8
#define HLO_MAX_EW_OPS 16

typedef enum {
  HLO_OK = 0,
  HLO_ERR_INVALID_ARG = 1, /* a constraint of the op's semantics or of this ABI is violated */
  HLO_ERR_UNSUPPORTED = 2, /* valid, but this library has no kernel for it (e.g. an element type) */
  HLO_ERR_CUDA = 3,        /* a CUDA call failed; the message carries cudaGetErrorString */
  HLO_ERR_WORKSPACE = 4    /* the workspace passed is smaller than hlo_reduce_workspace_size() */
} hlo_status;

/* Element types ("StableHLO Specification", section "Types"). */
typedef enum {
  HLO_F32 = 0,
  HLO_BF16 = 1,
  HLO_S8 = 2,
  HLO_F16 = 3,
  HLO_S32 = 4
} hlo_dtype;

/* A dense array: logical shape plus physical layout. */
typedef struct {
  int32_t rank;                            /* 0..HLO_MAX_RANK */
  int32_t dtype;                           /* hlo_dtype */
  int64_t dims[HLO_MAX_RANK];              /* dims[0..rank-1], each >= 0 */
  int64_t minor_to_major[HLO_MAX_RANK];    /* a permutation of 0..rank-1, minor-most first */
} hlo_array;

/* Elementwise ops of a prologue/epilogue chain. Each is the IEEE-754 operation on the element type
 * ("StableHLO Specification", sections "exponential", "log", "tanh", "abs", "negate", "add",
 * "multiply", "constant"); the result type equals the operand type (constraint C1 of each op). The
 * chain carries one running value v, which starts as the element x entering the chain:
 *   HLO_EW_EXP/LOG/TANH/ABS/NEG  v = op(v)
 *   HLO_EW_ADD_BCAST             v = v + broadcast_in_dim(bcast, bcast_dimensions)[i]
 *   HLO_EW_ADD_CONST/MUL_CONST   v = v + c, v * c, with c = imm[k] as a constant of the element type
 *                                (the double is rounded to the element type, nearest even)
 *   HLO_EW_ADD_INPUT/MUL_INPUT   v = v + x, v * x (x: the element that entered the chain)
 * So any expression that folds the input into one running value with constants is a chain; the GELU
 * loop fusion of "XLA:GPU Emitters" (section "Loop emitter") is
 *   MUL_INPUT, MUL_INPUT, MUL_CONST 0.044708, ADD_INPUT, MUL_CONST 0.79785, TANH, ADD_CONST 1,
 *   MUL_CONST 0.5, MUL_INPUT.
 * Rounding: exp, log and tanh are correctly rounded to the element type (f32, bf16, f16) and the other
 * ops are exact IEEE operations, with one exception: a reduce with the add body whose prologue is
 * exactly (exp) or (exp, add of a bf16 vector broadcast along the reduced dimension) evaluates that
 * exp with a faster approximation (relative error below about 2^-17). For f32 terms this stays inside
 * the reduction's tolerance for any input; a 16-bit term can come out one unit of its type away from
 * the correctly rounded one when exp lies that close to a rounding boundary (rare for spread-out
 * inputs; the tolerance holds for them, not for inputs made only of such values). */
typedef enum {
  HLO_EW_EXP = 1,
  HLO_EW_LOG = 2,
  HLO_EW_ABS = 3,
  HLO_EW_NEG = 4,
  HLO_EW_ADD_BCAST = 5, /* v + broadcast_in_dim(bcast, bcast_dimensions) */
  HLO_EW_TANH = 6,
  HLO_EW_ADD_CONST = 7,
  HLO_EW_MUL_CONST = 8,
  HLO_EW_ADD_INPUT = 9,
  HLO_EW_MUL_INPUT = 10
} hlo_ew_kind;

/* A chain of up to HLO_MAX_EW_OPS elementwise ops applied in order to every element of the array
 * it is attached to. n_ops == 0 (or a NULL chain pointer) is the identity.
 *
 * HLO_EW_ADD_BCAST adds broadcast_in_dim(bcast, bcast_dimensions) ("StableHLO Specification", section
 * "broadcast_in_dim"): the operand element read for array index i has, in each operand dimension d,
 * index 0 if bcast.dims[d] == 1 and i[bcast_dimensions[d]] otherwise (constraints C2-C5 are checked:
 * one entry per operand dimension, each in range and unique, and bcast.dims[d] is 1 or equal to the
 * array's dimension). bcast.dtype must equal the array's element type (add, constraint C1).
 *
 * round_intermediates selects the precision of values between ops for 16-bit float arrays:
 *   1 -- every op result is rounded to the element type (the spec's types: exp of bf16 is bf16);
 *   0 -- intermediates stay in f32 and only the hero sees them.
 * For f32 arrays the two are the same. */
typedef struct {
  int32_t n_ops;
  int32_t ops[HLO_MAX_EW_OPS];             /* hlo_ew_kind */
  int32_t round_intermediates;
  const void* bcast_ptr;                   /* device pointer; used by HLO_EW_ADD_BCAST only */
  hlo_array bcast;
  int64_t bcast_dimensions[HLO_MAX_RANK];
  double imm[HLO_MAX_EW_OPS];              /* the constant of op k (HLO_EW_ADD_CONST/MUL_CONST) */
} hlo_ew_chain;

typedef enum { HLO_RED_ADD = 0, HLO_RED_MAX = 1 } hlo_reduce_kind;

/* Uniform quantization parameters ("StableHLO Specification", section "Types", quantized element
 * types; "StableHLO Quantization", per-tensor and per-axis quantization):
 *   real = scale * (q - zero_point),
 * one (scale, zero_point) pair for the whole tensor (quantization_dimension = -1, n = 1) or one pair
 * per slice t[..., i, ...] along quantization_dimension (n = dims[quantization_dimension]).
 * scales / zero_points point to n values on the DEVICE. host_scales / host_zero_points optionally
 * point to a host copy of the same values: when given, the library checks the spec's constraints on
 * them (C6 scale > 0, C7 finite, C8 storage_min <= zero_point <= storage_max); when NULL those value
 * constraints are the caller's responsibility. For per-tensor parameters the host copy alone is
 * enough (the device pointers may then be NULL). storage_min < storage_max must lie within the
 * storage type's range (C4). */
typedef struct {
  int32_t quantization_dimension;          /* -1: per-tensor */
  int64_t n;
  const float* scales;                     /* device */
  const int32_t* zero_points;              /* device */
  const float* host_scales;                /* optional host copy */
  const int32_t* host_zero_points;         /* optional host copy */
  int32_t storage_min;
  int32_t storage_max;
} hlo_quant;

/* ------------------------------------------------------------------------------------------------
 * hlo_reduce_fusion -- out = reduce(prologue(in), init_value, dimensions, kind).
 *
 * Semantics: "StableHLO Specification", section "reduce" (inputs I1-I4, constraints C1-C8), with the
 * body add or maximum ("StableHLO Specification", section "maximum": IEEE-754 maximum, NaN propagates,
 * -0 < +0) and "XLA Operation Semantics", section "Reduce". Every output element is the reduction of
 * the prologue applied to its slice; init_value is applied exactly once. The dimensions kept form the
 * output in their original relative order (C7); out describes that shape with any layout.
 *
 *   in, in_ptr       input array (f32, bf16 or f16) and its device data
 *   prologue         elementwise chain applied to every input element first (may be NULL)
 *   dimensions       n_dimensions unique dimension numbers of in to reduce (C4, C5); may be 0 of them
 *   kind             HLO_RED_ADD or HLO_RED_MAX
 *   init_value       the init value, converted to the accumulation type
 *   accum_dtype      must be HLO_F32 (the body's element type; inputs are promoted to it, C6)
 *   out, out_ptr     output array (f32, bf16 or f16); the f32 result is rounded to nearest even
 *   workspace        device scratch of at least hlo_reduce_workspace_size() bytes, or NULL with
 *                    workspace_bytes == 0. The library only uses it for row reductions with too few
 *                    rows to occupy the device (for example a reduction of a whole array to one
 *                    value): each row is cut into segments that separate blocks reduce into the
 *                    workspace, and a second kernel combines every row's partials in segment order.
 *                    Without a workspace such reductions still run, unsplit, on as many blocks as there
 *                    are rows. A non-NULL workspace smaller than needed is HLO_ERR_WORKSPACE; one that
 *                    overlaps the input or output is HLO_ERR_INVALID_ARG. Its contents on entry do not
 *                    matter, and calls that share one workspace must not overlap in time.
 *
 * A reduced dimension of size 0 yields init_value. Reductions whose reduced dimensions are the
 * minor-most physical dimensions run as row reductions, those with kept dimensions on both sides
 * as column reductions (thread-block clusters combine row slabs through distributed shared memory);
 * any other pattern runs a general kernel.
 * ---------------------------------------------------------------------------------------------- */
hlo_status hlo_reduce_fusion(const hlo_array* in, const void* in_ptr, const hlo_ew_chain* prologue,
                             const int64_t* dimensions, int32_t n_dimensions, int32_t kind,
                             double init_value, int32_t accum_dtype, const hlo_array* out,
                             void* out_ptr, void* workspace, size_t workspace_bytes, void* stream);

/* Device scratch bytes hlo_reduce_fusion can use for this input and reduction on the current device:
 * 4 bytes per (row, segment) partial when the rows are split (see workspace above), else 0. Returns 0
 * for invalid arguments as well. */
size_t hlo_reduce_workspace_size(const hlo_array* in, const int64_t* dimensions, int32_t n_dimensions,
                                 int32_t accum_dtype);

/* ------------------------------------------------------------------------------------------------
 * hlo_reduce_fusion_noalloc -- hlo_reduce_fusion for callers that cannot allocate device memory.
 *
 * No counterpart in the pages: this is a convenience of the library. Some callers cannot allocate a
 * device workspace where they run a reduction -- for example code embedded in another runtime that owns
 * all device memory through its own allocator, or code held to a memory budget fixed when it started.
 * This entry point takes the same arguments as hlo_reduce_fusion without the workspace, allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine), and computes the same result: when
 * the reduction splits its rows (see hlo_reduce_fusion's workspace), the partials go to a scratch array
 * of 64 KiB that the library keeps in device memory on every device that loads it, until the process
 * exits.
 *   - A reduction that needs more than 64 KiB of scratch (hlo_reduce_workspace_size) is rejected with
 *     HLO_ERR_WORKSPACE and a message; on this library's current plans that takes a device with far
 *     more than 2000 SMs.
 *   - The first call on a device that needs the scratch looks up its device address
 *     (cudaGetSymbolAddress), once per device, with that device current; make that first call before
 *     any stream capture.
 *   - Every call on a device shares the one array. Nothing in it has to start at zero (each call
 *     writes every partial before reading it), but calls whose kernels overlap on the GPU -- on
 *     different streams, or from different host threads -- race on it and must be serialised.
 * ---------------------------------------------------------------------------------------------- */
hlo_status hlo_reduce_fusion_noalloc(const hlo_array* in, const void* in_ptr, const hlo_ew_chain* prologue,
                                     const int64_t* dimensions, int32_t n_dimensions, int32_t kind,
                                     double init_value, int32_t accum_dtype, const hlo_array* out, void* out_ptr,
                                     void* stream);

/* ------------------------------------------------------------------------------------------------
 * hlo_transpose_fusion -- out = epilogue(transpose(prologue(in), permutation)), or with
 * self_add_epilogue != 0: out = epilogue(prologue(in) + transpose(prologue(in), permutation)).
 *
 * Semantics: transpose maps output index r to input index i with i[permutation[k]] = r[k], so
 * dims(out)[k] = dims(in)[permutation[k]] -- the output-to-input indexing map of "XLA:GPU Emitters",
 * section "Indexing transformations" ([20,40] -> [40,20] reads (d0, d1) -> (d1, d0)). The self-add form
 * is the fusion of "XLA:GPU Emitters", section "Partitioning": log(param) feeding both a transpose and
 * an add; it requires dims(out) == dims(in). Its prologue is evaluated once per input element (the
 * kernel loads the tile pair (I,J), (J,I) once and reuses both), and add is the IEEE f32 add, so the
 * result is bitwise symmetric for a 2-D square input.
 *
 *   in, in_ptr       input array; element types f32, bf16, f16 (with chains) or any (no chains)
 *   prologue         chain applied to the input elements (may be NULL)
 *   permutation      rank entries, a permutation of 0..rank-1
 *   epilogue         chain applied to the output elements (may be NULL; no HLO_EW_ADD_BCAST)
 *   out, out_ptr     output array: same element type, dims as above, any layout
 * ---------------------------------------------------------------------------------------------- */
hlo_status hlo_transpose_fusion(const hlo_array* in, const void* in_ptr, const hlo_ew_chain* prologue,
                                const int64_t* permutation, int32_t self_add_epilogue,
                                const hlo_ew_chain* epilogue, const hlo_array* out, void* out_ptr,
                                void* stream);

/* ------------------------------------------------------------------------------------------------
 * hlo_layout_convert -- the same logical array written with another minor_to_major ("XLA Shapes and
 * Layout", section "Layout"): for every index i, out[offset(i, out_minor_to_major)] =
 * in[offset(i, in->minor_to_major)]. Any element type; bit-exact.
 *   out_minor_to_major   in->rank entries, a permutation of 0..rank-1
 * ---------------------------------------------------------------------------------------------- */
hlo_status hlo_layout_convert(const hlo_array* in, const void* in_ptr, const int64_t* out_minor_to_major,
                              void* out_ptr, void* stream);

/* ------------------------------------------------------------------------------------------------
 * hlo_quant_fusion -- dequantize -> elementwise float ops -> layout change -> quantize.
 *
 *   real = scale[j] * (q - zero_point[j])                       (f32: exact difference, one rounding)
 *   real = float_ops(real)                                      (f32 chain, may be NULL)
 *   out  = clamp(round_nearest_even(real / out_scale[j']) + out_zero_point[j'],
 *                storage_min, storage_max)                      (f32 IEEE division)
 * with j / j' the index along the input / output quantization_dimension (0 per-tensor). This is the
 * dequantize -> float op -> quantize pattern of "StableHLO Quantization" (quantized ops expressed as
 * dequantize_op_quantize) with the relation real = scale * (q - zero_point); rounding is
 * roundToIntegralTiesToEven ("StableHLO Specification", section "round_nearest_even") and saturation is
 * clamp ("StableHLO Specification", section "clamp"). With out_q == NULL the output is the f32 real.
 *
 *   in, in_ptr           storage array, dtype HLO_S8
 *   in_q                 its quantization parameters (required)
 *   float_ops            f32 chain applied to the dequantized values (may be NULL)
 *   out_minor_to_major   output layout (rank entries); must equal out->minor_to_major
 *   out, out_ptr         output array: dims equal to in's, dtype HLO_S8 (quantized) or HLO_F32
 *   out_q                output quantization parameters, or NULL for f32 output
 * Bit-exact: both the dequantize product and the quantize division are single IEEE f32 operations.
 * ---------------------------------------------------------------------------------------------- */
hlo_status hlo_quant_fusion(const hlo_array* in, const void* in_ptr, const hlo_quant* in_q,
                            const hlo_ew_chain* float_ops, const int64_t* out_minor_to_major,
                            const hlo_array* out, void* out_ptr, const hlo_quant* out_q, void* stream);

/* ------------------------------------------------------------------------------------------------
 * Elementwise binary op on per-tensor quantized operands ("StableHLO Specification", sections "add",
 * "divide", "maximum", "minimum", "multiply": for quantized types each performs
 * dequantize_op_quantize(op, lhs, rhs, type(result))):
 *     out[i] = clamp(round_nearest_even(op(dl, dr) / s_out) + zp_out, storage_min, storage_max)
 *     dl = s_l * (lhs[i] - zp_l),  dr = s_r * (rhs[i] - zp_r)
 * with every float step a single IEEE f32 operation (maximum/minimum propagate NaN; a NaN result
 * quantizes to zp_out), so the result is bit-exact.
 *   op                    HLO_QOP_ADD, HLO_QOP_DIVIDE, HLO_QOP_MAXIMUM, HLO_QOP_MINIMUM, HLO_QOP_MULTIPLY
 *   lhs, rhs, out         HLO_S8 arrays with equal dims, any layouts (element i is the same logical
 *                         index in each)
 *   lhs_q, rhs_q, out_q   per-tensor parameters (quantization_dimension -1, host_scales and
 *                         host_zero_points set); per-axis operands are rejected (I1, I2 of each op)
 * ---------------------------------------------------------------------------------------------- */
typedef enum {
  HLO_QOP_ADD = 0,
  HLO_QOP_DIVIDE = 1,
  HLO_QOP_MAXIMUM = 2,
  HLO_QOP_MINIMUM = 3,
  HLO_QOP_MULTIPLY = 4
} hlo_quant_binary_op;

hlo_status hlo_quant_binary(int32_t op, const hlo_array* lhs, const void* lhs_ptr, const hlo_quant* lhs_q,
                            const hlo_array* rhs, const void* rhs_ptr, const hlo_quant* rhs_q, const hlo_array* out,
                            void* out_ptr, const hlo_quant* out_q, void* stream);

/* ------------------------------------------------------------------------------------------------
 * Data movement of quantized tensors. Stored codes move like plain elements (result[result_index] =
 * operand[operand_index]); the result's quantization parameters follow the ops' quantized constraints.
 * Note: add, divide, maximum, minimum and multiply take per-tensor quantized operands only (inputs I1,
 * I2 of each op), which is why hlo_quant_binary rejects per-axis ones; per-axis tensors are moved by the
 * two entry points below.
 *
 * hlo_quant_broadcast_in_dim ("StableHLO Specification", section "broadcast_in_dim", constraints C1-C6):
 *   operand, operand_ptr, operand_q   HLO_S8 operand and its parameters (per-tensor or per-axis)
 *   broadcast_dimensions              operand->rank entries: result dimension of each operand dimension
 *                                     (C3 in range, C4 unique, C5 size 1 or equal)
 *   result, result_ptr                HLO_S8 result (any layout)
 *   result_quantization_dimension     (host, out) -1 for a per-tensor operand; otherwise
 *                                     broadcast_dimensions[quantization_dimension(operand)] (C6)
 *   result_scales, result_zero_points (device, out) the result's pairs: 1 for per-tensor; otherwise
 *                                     dim(result, *result_quantization_dimension) pairs, the operand's,
 *                                     or its single pair repeated when dim(operand, qd) = 1 (C6)
 *
 * hlo_quant_reshape ("StableHLO Specification", section "reshape", constraints C1-C3): the element at
 * lexicographic position p of the operand becomes the element at position p of the result, in each
 * array's own layout (bit-exact, any element type).
 *   operand_q                       NULL for an unquantized array; else the operand's parameters (HLO_S8)
 *   result_quantization_dimension   the result type's quantization dimension: -1 for unquantized and
 *                                   per-tensor operands; for a per-axis operand a result dimension with
 *                                   the same size and the same products of the dimensions before and
 *                                   after it (C3), HLO_ERR_INVALID_ARG otherwise. The (scale,
 *                                   zero_point) pairs are the operand's, unchanged (C1).
 * ---------------------------------------------------------------------------------------------- */
hlo_status hlo_quant_broadcast_in_dim(const hlo_array* operand, const void* operand_ptr, const hlo_quant* operand_q,
                                      const int64_t* broadcast_dimensions, const hlo_array* result, void* result_ptr,
                                      float* result_scales, int32_t* result_zero_points,
                                      int32_t* result_quantization_dimension, void* stream);
hlo_status hlo_quant_reshape(const hlo_array* operand, const void* operand_ptr, const hlo_quant* operand_q,
                             const hlo_array* result, int32_t result_quantization_dimension, void* result_ptr,
                             void* stream);

/* ------------------------------------------------------------------------------------------------
 * Variadic reduce with the max/argmax body ("XLA Operation Semantics", section "Variadic Reduce"):
 * inputs V and K, init values I_V, I_K, and the body
 *     f(max, argmax, value, index) = (value, index) if value >= max else (max, argmax)
 * applied from f(I_V, I_K, V_0, K_0) on, along the lexicographic walk of the reduced dimensions (in
 * increasing dimension order). So equal maxima keep the last index walked, and NaN values are never
 * selected (a comparison with NaN is false). The result is exact: a member of V (or I_V) and of K
 * (or I_K).
 *
 *   in, in_ptr          V: float element type (HLO_F32, HLO_BF16, HLO_F16), any layout
 *   idx, idx_ptr        K: HLO_S32, same dims as V, any layout; or idx_ptr == NULL, then K is the
 *                       position along the reduced dimension (n_dimensions must be 1: the iota of
 *                       the pages' example)
 *   dimensions          n_dimensions distinct dimensions of V to reduce (may be 0)
 *   init_value          I_V, rounded to V's element type (nearest even)
 *   init_index          I_K, in the s32 range
 *   out, out_ptr        the maxima: V's element type, dims = V's kept dims in order, any layout
 *   out_idx, out_idx_ptr the indices: HLO_S32, same dims as out, any layout
 * Errors as for hlo_reduce_fusion (C4, C5, C7 of "reduce"); buffers must not overlap the outputs.
 * ---------------------------------------------------------------------------------------------- */
hlo_status hlo_reduce_max_argmax(const hlo_array* in, const void* in_ptr, const hlo_array* idx,
                                 const void* idx_ptr, const int64_t* dimensions, int32_t n_dimensions,
                                 double init_value, int64_t init_index, const hlo_array* out, void* out_ptr,
                                 const hlo_array* out_idx, void* out_idx_ptr, void* stream);

/* ------------------------------------------------------------------------------------------------
 * Device-side faults. A kernel that gives up on a bounded wait records a fault bit in a word the
 * library keeps on each device (no counterpart in the pages: this is the library's own diagnostics).
 *   HLO_FAULT_COPY_TIMEOUT  a kernel that streams tiles through shared memory (the streaming row
 *                           reduce, the tensor-copy transposes, the quantized relayout, the generated
 *                           chain kernels) waited about one second for an asynchronous global -> shared
 *                           copy without seeing it complete; that block stopped, waited (again with a
 *                           bound) for its copies in flight and returned without writing the rest of
 *                           its outputs (the streaming row reduce writes NaN to its rows), so the
 *                           launch itself still reports success.
 *
 * hlo_device_faults waits for all work on the current device (cudaDeviceSynchronize), then stores the
 * fault bits recorded there since the last clear, by any of the library's kernels, in *faults (0: none)
 * and, if clear != 0, resets them.
 * HLO_ERR_CUDA if the device reports an error.
 *
 * hlo_selftest_bounded_wait enqueues one block that waits, bounded to about a millisecond, on a barrier
 * nothing completes, and records HLO_FAULT_COPY_TIMEOUT as the streaming kernel would: it checks the
 * reporting path without a failing copy.
 * ---------------------------------------------------------------------------------------------- */
#define HLO_FAULT_COPY_TIMEOUT 1u

hlo_status hlo_device_faults(uint32_t* faults, int32_t clear);
hlo_status hlo_selftest_bounded_wait(void* stream);

/* ------------------------------------------------------------------------------------------------
 * Generated chain kernels ("XLA:GPU Emitters", section "Loop emitter": one kernel is emitted per
 * fusion, its elementwise ops as straight-line code). For an identity-layout transpose fusion on
 * bf16 / f16 of 2^20 elements or more, 16-byte aligned, whose prologue rounds every op to the element
 * type and uses only add / multiply by the input or a constant, negate, absolute value and (bf16)
 * tanh, hlo_transpose_fusion writes the chain as CUDA source, compiles it once per device with NVRTC
 * (opened with dlopen on first use) and launches the result; the results are the bits the library's
 * other kernels give. If NVRTC cannot be opened or the source does not compile, the library's fixed
 * kernels run the call instead.
 *
 * When a bf16 chain's tanh ops all lie in one run of two or more ops that do not read the input (for
 * GELU: multiply by a constant, tanh, add 1, multiply by 1/2), the first call also builds that run's
 * 65536-entry result table on the device, on the call's stream, into one of eight slots the library
 * holds for the life of the process (later such chains use the tanh table instead); calls on other
 * streams wait for it with cudaStreamWaitEvent. While the call's stream is being captured into a CUDA
 * graph, only a chain compiled earlier and without such a table uses its generated kernel: nothing is
 * compiled, built or waited for inside a capture.
 *
 * hlo_jit_kernels returns the number of chain kernels built so far for the current device, or -1 when
 * NVRTC or the driver calls it needs are unavailable (no generated kernels will run).
 *
 * hlo_jit_source writes the CUDA C source the library generates for `chain` on element type `dtype`
 * (HLO_BF16 or HLO_F16) into buf, NUL-terminated, when buf_len exceeds its length; it returns the
 * length (without the NUL), or -1 when the generator does not take the chain (another element type,
 * intermediates not rounded, an op other than those above) or buf_len < 0, or buf is NULL with
 * buf_len > 0. With buf NULL and buf_len 0 it only measures. The source is the one generated while a
 * run-table slot is free. No device, NVRTC or driver call is made; the caller owns buf.
 * ---------------------------------------------------------------------------------------------- */
int32_t hlo_jit_kernels(void);
int64_t hlo_jit_source(const hlo_ew_chain* chain, int32_t dtype, char* buf, int64_t buf_len);

/* ------------------------------------------------------------------------------------------------
 * Fault injection for tests of the error path (no counterpart in the pages: the library's own test
 * support). When the environment variable HLOFUSION_FAULT holds an entry point's name (for example
 * "hlo_transpose_fusion") or "all", that entry point validates its arguments as usual and then returns
 * HLO_ERR_CUDA, with "injected fault" in hlo_last_error(), before it enqueues any work. Calls that fail
 * validation still report their own error. The variable is read on every call; unset or empty, nothing
 * changes.
 * ---------------------------------------------------------------------------------------------- */

/* Thread-local description of the last error returned on this thread ("" if none). */
const char* hlo_last_error(void);

/* Library version string. */
const char* hlo_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HLO_FUSION_H */
