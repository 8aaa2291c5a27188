"""transpose_heroes_gb300 -- HLO reduce / transpose / layout / quantized-relayout hero fusions on GB300.

Thin Python binding over the C ABI of libhlofusion (include/hlo_fusion.h). Each function marshals its
arguments into the C descriptors and calls the entry point of the same name; every step of the fusion
runs in the library's CUDA kernels. PyTorch only supplies device memory and the current stream.

Arrays are passed as device tensors holding the PHYSICAL buffer (any torch dtype of the right element
size; flat is simplest) together with a description: dims, minor_to_major and the element type name
("f32", "bf16", "f16", "s8", "s32"). There is no CPU fallback: if the library is not built, or no CUDA
device is present, the calls raise.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libhlofusion.so")

MAX_RANK = 8
MAX_EW_OPS = 16
DTYPES = {"f32": 0, "bf16": 1, "s8": 2, "f16": 3, "s32": 4}
OPS = {"exp": 1, "log": 2, "abs": 3, "neg": 4, "add_bcast": 5, "tanh": 6, "add_const": 7, "mul_const": 8,
       "add_input": 9, "mul_input": 10}
REDUCE_KINDS = {"add": 0, "max": 1}
STATUS_INVALID_ARG = 1
STATUS = {0: "HLO_OK", 1: "HLO_ERR_INVALID_ARG", 2: "HLO_ERR_UNSUPPORTED", 3: "HLO_ERR_CUDA", 4: "HLO_ERR_WORKSPACE"}

# Every function the header declares; the library must export all of them.
EXPORTS = ("hlo_reduce_fusion", "hlo_reduce_fusion_noalloc", "hlo_reduce_workspace_size", "hlo_transpose_fusion",
           "hlo_layout_convert",
           "hlo_quant_fusion", "hlo_quant_binary", "hlo_quant_broadcast_in_dim", "hlo_quant_reshape",
           "hlo_reduce_max_argmax", "hlo_device_faults",
           "hlo_selftest_bounded_wait", "hlo_jit_kernels", "hlo_jit_source", "hlo_last_error", "hlo_version")
QUANT_BINARY_OPS = {"add": 0, "divide": 1, "maximum": 2, "minimum": 3, "multiply": 4}


class HloError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class Array(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("dims", ctypes.c_int64 * MAX_RANK), ("minor_to_major", ctypes.c_int64 * MAX_RANK)]


class EwChain(ctypes.Structure):
    _fields_ = [("n_ops", ctypes.c_int32), ("ops", ctypes.c_int32 * MAX_EW_OPS),
                ("round_intermediates", ctypes.c_int32), ("bcast_ptr", ctypes.c_void_p),
                ("bcast", Array), ("bcast_dimensions", ctypes.c_int64 * MAX_RANK),
                ("imm", ctypes.c_double * MAX_EW_OPS)]


class Quant(ctypes.Structure):
    _fields_ = [("quantization_dimension", ctypes.c_int32), ("n", ctypes.c_int64),
                ("scales", ctypes.c_void_p), ("zero_points", ctypes.c_void_p),
                ("host_scales", ctypes.c_void_p), ("host_zero_points", ctypes.c_void_p),
                ("storage_min", ctypes.c_int32), ("storage_max", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return LIB_PATH


def lib() -> ctypes.CDLL:
    """Loads libhlofusion.so (built by build.py / __graft_entry__.build()). Raises if missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libhlofusion.so is not built ({LIB_PATH}); run transpose_heroes_gb300.build.build()")
            h = ctypes.CDLL(LIB_PATH)
            P = ctypes.POINTER
            vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
            h.hlo_reduce_fusion.argtypes = [P(Array), vp, P(EwChain), P(i64), i32, i32, ctypes.c_double, i32,
                                            P(Array), vp, vp, ctypes.c_size_t, vp]
            h.hlo_reduce_fusion.restype = ctypes.c_int
            h.hlo_reduce_fusion_noalloc.argtypes = [P(Array), vp, P(EwChain), P(i64), i32, i32, ctypes.c_double, i32,
                                                    P(Array), vp, vp]
            h.hlo_reduce_fusion_noalloc.restype = ctypes.c_int
            h.hlo_reduce_workspace_size.argtypes = [P(Array), P(i64), i32, i32]
            h.hlo_reduce_workspace_size.restype = ctypes.c_size_t
            h.hlo_transpose_fusion.argtypes = [P(Array), vp, P(EwChain), P(i64), i32, P(EwChain), P(Array), vp, vp]
            h.hlo_transpose_fusion.restype = ctypes.c_int
            h.hlo_layout_convert.argtypes = [P(Array), vp, P(i64), vp, vp]
            h.hlo_layout_convert.restype = ctypes.c_int
            h.hlo_quant_fusion.argtypes = [P(Array), vp, P(Quant), P(EwChain), P(i64), P(Array), vp, P(Quant), vp]
            h.hlo_quant_fusion.restype = ctypes.c_int
            h.hlo_quant_binary.argtypes = [i32, P(Array), vp, P(Quant), P(Array), vp, P(Quant), P(Array), vp,
                                           P(Quant), vp]
            h.hlo_quant_binary.restype = ctypes.c_int
            h.hlo_reduce_max_argmax.argtypes = [P(Array), vp, P(Array), vp, P(i64), i32, ctypes.c_double, i64,
                                                P(Array), vp, P(Array), vp, vp]
            h.hlo_reduce_max_argmax.restype = ctypes.c_int
            h.hlo_quant_broadcast_in_dim.argtypes = [P(Array), vp, P(Quant), P(i64), P(Array), vp, vp, vp,
                                                     P(ctypes.c_int32), vp]
            h.hlo_quant_broadcast_in_dim.restype = ctypes.c_int
            h.hlo_quant_reshape.argtypes = [P(Array), vp, P(Quant), P(Array), i32, vp, vp]
            h.hlo_quant_reshape.restype = ctypes.c_int
            h.hlo_device_faults.argtypes = [P(ctypes.c_uint32), i32]
            h.hlo_device_faults.restype = ctypes.c_int
            h.hlo_selftest_bounded_wait.argtypes = [vp]
            h.hlo_selftest_bounded_wait.restype = ctypes.c_int
            h.hlo_jit_kernels.argtypes = []
            h.hlo_jit_kernels.restype = ctypes.c_int32
            h.hlo_jit_source.argtypes = [P(EwChain), i32, ctypes.c_char_p, i64]
            h.hlo_jit_source.restype = ctypes.c_int64
            h.hlo_last_error.restype = ctypes.c_char_p
            h.hlo_version.restype = ctypes.c_char_p
            _lib = h
    return _lib


def last_error() -> str:
    return lib().hlo_last_error().decode()


def version() -> str:
    return lib().hlo_version().decode()


# ---- marshalling helpers ---------------------------------------------------------------------------
def default_m2m(rank: int):
    return list(range(rank - 1, -1, -1))


def make_array(dims: Sequence[int], m2m: Optional[Sequence[int]], dtype: str) -> Array:
    dims = [int(d) for d in dims]
    m2m = default_m2m(len(dims)) if m2m is None else [int(d) for d in m2m]
    a = Array()
    a.rank = len(dims)
    a.dtype = DTYPES[dtype]
    for i, d in enumerate(dims):
        a.dims[i] = d
    for i, d in enumerate(m2m):
        a.minor_to_major[i] = d
    return a


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _i64(values):
    values = [int(v) for v in values]
    return (ctypes.c_int64 * max(1, len(values)))(*values)


def _stream(stream) -> int:
    if stream is None:
        import torch

        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def make_chain(spec) -> Optional[EwChain]:
    """spec: {"ops": [...], "round_each": bool, "bcast": {"tensor", "dims", "m2m", "dtype",
    "broadcast_dimensions"}} or None. An op is a name, or (name, constant) for add_const/mul_const."""
    if spec is None or not spec.get("ops"):
        return None
    c = EwChain()
    ops = list(spec["ops"])
    if len(ops) > MAX_EW_OPS:
        raise HloError(STATUS_INVALID_ARG, f"a chain holds at most {MAX_EW_OPS} ops")
    c.n_ops = len(ops)
    for i, op in enumerate(ops):
        if isinstance(op, (tuple, list)):
            op, c.imm[i] = op[0], float(op[1])
        c.ops[i] = OPS[op]
    c.round_intermediates = 1 if spec.get("round_each", True) else 0
    b = spec.get("bcast")
    if b is not None:
        c.bcast_ptr = _ptr(b["tensor"])
        c.bcast = make_array(b["dims"], b.get("m2m"), b["dtype"])
        for i, d in enumerate(b["broadcast_dimensions"]):
            c.bcast_dimensions[i] = int(d)
    return c


class _QuantKeep:
    def __init__(self, spec):
        self.keep = []
        self.q = None
        if spec is None:
            return
        q = Quant()
        qd = spec.get("quantization_dimension")
        q.quantization_dimension = -1 if qd is None else int(qd)
        hs = spec.get("host_scales")
        hz = spec.get("host_zero_points")
        n = spec.get("n")
        if hs is not None:
            hs = np.ascontiguousarray(np.atleast_1d(hs), dtype=np.float32)
            hz = np.ascontiguousarray(np.atleast_1d(hz), dtype=np.int32)
            self.keep += [hs, hz]
            q.host_scales = hs.ctypes.data
            q.host_zero_points = hz.ctypes.data
            n = hs.size if n is None else n
        q.n = int(n if n is not None else spec["scales"].numel())
        # device parameters (per-axis); host arrays under these keys are not device memory
        dev = lambda t: _ptr(t) if t is not None and not isinstance(t, np.ndarray) else 0
        q.scales = dev(spec.get("scales"))
        q.zero_points = dev(spec.get("zero_points"))
        q.storage_min = int(spec.get("storage_min", -128))
        q.storage_max = int(spec.get("storage_max", 127))
        self.q = q

    def ref(self):
        return None if self.q is None else ctypes.byref(self.q)


def _check(status: int):
    if status != 0:
        raise HloError(status, last_error())


def _ref(x):
    return None if x is None else ctypes.byref(x)


# ---- entry points ------------------------------------------------------------------------------------
def reduce_fusion(inp, in_dims, in_dtype, dimensions, kind, init, out, out_dtype, in_m2m=None, out_m2m=None,
                  prologue=None, workspace=None, workspace_bytes=0, stream=None):
    """hlo_reduce_fusion: out = reduce(prologue(inp), init, dimensions, kind) with f32 accumulation."""
    a = make_array(in_dims, in_m2m, in_dtype)
    red = set(int(d) for d in dimensions)
    out_dims = [d for i, d in enumerate(in_dims) if i not in red]
    o = make_array(out_dims, out_m2m, out_dtype)
    ch = make_chain(prologue)
    dims = _i64(dimensions)
    _check(lib().hlo_reduce_fusion(ctypes.byref(a), _ptr(inp), _ref(ch), dims, len(list(dimensions)),
                                   REDUCE_KINDS[kind], float(init), DTYPES["f32"], ctypes.byref(o), _ptr(out),
                                   _ptr(workspace), int(workspace_bytes), _stream(stream)))
    return out


def reduce_fusion_noalloc(inp, in_dims, in_dtype, dimensions, kind, init, out, out_dtype, in_m2m=None, out_m2m=None,
                          prologue=None, stream=None):
    """hlo_reduce_fusion_noalloc: the same reduce with no workspace argument, for callers that cannot
    allocate device memory; split rows use the library's own 64 KiB scratch on the device."""
    a = make_array(in_dims, in_m2m, in_dtype)
    red = set(int(d) for d in dimensions)
    out_dims = [d for i, d in enumerate(in_dims) if i not in red]
    o = make_array(out_dims, out_m2m, out_dtype)
    ch = make_chain(prologue)
    _check(lib().hlo_reduce_fusion_noalloc(ctypes.byref(a), _ptr(inp), _ref(ch), _i64(dimensions),
                                           len(list(dimensions)), REDUCE_KINDS[kind], float(init), DTYPES["f32"],
                                           ctypes.byref(o), _ptr(out), _stream(stream)))
    return out


def reduce_max_argmax(inp, in_dims, in_dtype, dimensions, out, out_idx, init_value=float("-inf"), init_index=-1,
                      indices=None, in_m2m=None, idx_m2m=None, out_m2m=None, out_idx_m2m=None, stream=None):
    """hlo_reduce_max_argmax: (out, out_idx) = variadic reduce of (inp, indices or the position along the
    single reduced dimension) with the max/argmax body; equal maxima keep the last index."""
    a = make_array(in_dims, in_m2m, in_dtype)
    red = set(int(d) for d in dimensions)
    out_dims = [d for i, d in enumerate(in_dims) if i not in red]
    o = make_array(out_dims, out_m2m, in_dtype)
    oi = make_array(out_dims, out_idx_m2m, "s32")
    k = make_array(in_dims, idx_m2m if idx_m2m is not None else in_m2m, "s32") if indices is not None else None
    _check(lib().hlo_reduce_max_argmax(ctypes.byref(a), _ptr(inp), _ref(k), _ptr(indices), _i64(dimensions),
                                       len(list(dimensions)), float(init_value), int(init_index), ctypes.byref(o),
                                       _ptr(out), ctypes.byref(oi), _ptr(out_idx), _stream(stream)))
    return out, out_idx


def quant_broadcast_in_dim(inp, dims, q, broadcast_dimensions, out, out_dims, out_scales, out_zero_points,
                           in_m2m=None, out_m2m=None, stream=None) -> int:
    """hlo_quant_broadcast_in_dim on s8 codes; writes the result's parameters into out_scales /
    out_zero_points (device tensors) and returns the result's quantization dimension (-1 per-tensor)."""
    a, o = make_array(dims, in_m2m, "s8"), make_array(out_dims, out_m2m, "s8")
    qk = _QuantKeep(q)
    rqd = ctypes.c_int32(0)
    _check(lib().hlo_quant_broadcast_in_dim(ctypes.byref(a), _ptr(inp), qk.ref(), _i64(broadcast_dimensions),
                                            ctypes.byref(o), _ptr(out), _ptr(out_scales), _ptr(out_zero_points),
                                            ctypes.byref(rqd), _stream(stream)))
    return int(rqd.value)


def reshape(inp, dims, out, out_dims, dtype, q=None, result_qdim=-1, in_m2m=None, out_m2m=None, stream=None):
    """hlo_quant_reshape: the lexicographic order is kept; q / result_qdim for quantized (s8) operands."""
    a, o = make_array(dims, in_m2m, dtype), make_array(out_dims, out_m2m, dtype)
    qk = _QuantKeep(q)
    _check(lib().hlo_quant_reshape(ctypes.byref(a), _ptr(inp), qk.ref(), ctypes.byref(o), int(result_qdim), _ptr(out),
                                   _stream(stream)))
    return out


FAULT_COPY_TIMEOUT = 1


def device_faults(clear: bool = False) -> int:
    """hlo_device_faults: the fault bits kernels recorded on the current device (waits for the device)."""
    f = ctypes.c_uint32(0)
    _check(lib().hlo_device_faults(ctypes.byref(f), 1 if clear else 0))
    return int(f.value)


def jit_kernels() -> int:
    """hlo_jit_kernels: chain kernels generated for the current device (-1: NVRTC unavailable)."""
    return int(lib().hlo_jit_kernels())


def jit_source(prologue, dtype: str):
    """hlo_jit_source: the CUDA source generated for a 16-bit chain, or None if the generator does not
    take it. `prologue` is a chain spec as for transpose_fusion."""
    chain = make_chain(prologue)
    if chain is None:
        return None
    n = int(lib().hlo_jit_source(ctypes.byref(chain), DTYPES[dtype], None, 0))
    if n < 0:
        return None
    buf = ctypes.create_string_buffer(n + 1)
    if int(lib().hlo_jit_source(ctypes.byref(chain), DTYPES[dtype], buf, n + 1)) != n:
        return None
    return buf.value.decode()


def selftest_bounded_wait(stream=None) -> None:
    """hlo_selftest_bounded_wait: one block's bounded wait runs out and records FAULT_COPY_TIMEOUT."""
    _check(lib().hlo_selftest_bounded_wait(_stream(stream)))


def reduce_workspace_size(in_dims, in_dtype, dimensions, in_m2m=None) -> int:
    a = make_array(in_dims, in_m2m, in_dtype)
    return int(lib().hlo_reduce_workspace_size(ctypes.byref(a), _i64(dimensions), len(list(dimensions)),
                                               DTYPES["f32"]))


def transpose_fusion(inp, in_dims, dtype, permutation, out, in_m2m=None, out_m2m=None, prologue=None,
                     self_add=False, epilogue=None, stream=None):
    """hlo_transpose_fusion: out = epilogue(T(prologue(inp))) or epilogue(f(inp) + T(f(inp)))."""
    a = make_array(in_dims, in_m2m, dtype)
    out_dims = [in_dims[p] for p in permutation]
    o = make_array(out_dims, out_m2m, dtype)
    pro, epi = make_chain(prologue), make_chain(epilogue)
    _check(lib().hlo_transpose_fusion(ctypes.byref(a), _ptr(inp), _ref(pro), _i64(permutation),
                                      1 if self_add else 0, _ref(epi), ctypes.byref(o), _ptr(out), _stream(stream)))
    return out


def layout_convert(inp, dims, dtype, in_m2m, out_m2m, out, stream=None):
    """hlo_layout_convert: the same logical array written with out_m2m."""
    a = make_array(dims, in_m2m, dtype)
    _check(lib().hlo_layout_convert(ctypes.byref(a), _ptr(inp), _i64(out_m2m), _ptr(out), _stream(stream)))
    return out


def quant_binary(op, lhs, rhs, dims, lhs_q, rhs_q, out, out_q, lhs_m2m=None, rhs_m2m=None, out_m2m=None,
                 stream=None):
    """hlo_quant_binary: out = quantize(op(dequantize(lhs), dequantize(rhs))), per-tensor s8 operands.
    The *_q specs carry host_scales / host_zero_points (one each)."""
    a, b, o = make_array(dims, lhs_m2m, "s8"), make_array(dims, rhs_m2m, "s8"), make_array(dims, out_m2m, "s8")
    ql, qr, qo = _QuantKeep(lhs_q), _QuantKeep(rhs_q), _QuantKeep(out_q)
    _check(lib().hlo_quant_binary(QUANT_BINARY_OPS[op], ctypes.byref(a), _ptr(lhs), ql.ref(), ctypes.byref(b), _ptr(rhs),
                                  qr.ref(), ctypes.byref(o), _ptr(out), qo.ref(), _stream(stream)))
    return out


def quant_fusion(inp, dims, in_q, out_m2m, out, out_dtype="s8", out_q=None, in_m2m=None, float_ops=None,
                 stream=None):
    """hlo_quant_fusion: dequantize -> float ops -> relayout -> quantize (or f32 output)."""
    a = make_array(dims, in_m2m, "s8")
    o = make_array(dims, out_m2m, out_dtype)
    qi, qo = _QuantKeep(in_q), _QuantKeep(out_q)
    ch = make_chain(float_ops)
    _check(lib().hlo_quant_fusion(ctypes.byref(a), _ptr(inp), qi.ref(), _ref(ch), _i64(out_m2m), ctypes.byref(o),
                                  _ptr(out), qo.ref(), _stream(stream)))
    return out
