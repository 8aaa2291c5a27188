"""Python access to the plain CPU oracle in ``oracle.cc``.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline are the only callers. The product library never imports this package, and this package
never imports the product. Arrays cross the boundary as flat numpy buffers in their PHYSICAL order
(the order the layout's minor_to_major gives), with the logical shape, the layout and the element
type passed alongside, exactly as a device buffer would be described.

Element types are named "f32", "bf16", "f16", "f64", "s8", "u8", "s32"; 16-bit floats are carried as
numpy uint16 arrays holding the raw bits.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cc")
_SO = os.path.join(_HERE, "liboracle.so")

MAX_RANK = 8
MAX_OPS = 16
DTYPES = {"f32": 0, "bf16": 1, "s8": 2, "f16": 3, "s32": 4, "f64": 5, "u8": 6}
NP_DTYPES = {"f32": np.float32, "bf16": np.uint16, "s8": np.int8, "f16": np.uint16,
             "s32": np.int32, "f64": np.float64, "u8": np.uint8}
OPS = {"exp": 1, "log": 2, "abs": 3, "neg": 4, "add_bcast": 5, "tanh": 6, "add_const": 7, "mul_const": 8,
       "add_input": 9, "mul_input": 10}
REDUCE_KINDS = {"add": 0, "max": 1}

# Compiler flags: no fast-math and no FMA contraction, so every source operation rounds exactly once.
CXXFLAGS = ["-O2", "-std=c++17", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile oracle.cc into liboracle.so next to it (g++, no CUDA). Returns the library path."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", *CXXFLAGS, _SRC, "-o", tmp])
        os.replace(tmp, _SO)
    return _SO


class Arr(ctypes.Structure):
    _fields_ = [("rank", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("dims", ctypes.c_int64 * MAX_RANK), ("m2m", ctypes.c_int64 * MAX_RANK)]


class Chain(ctypes.Structure):
    _fields_ = [("n_ops", ctypes.c_int32), ("ops", ctypes.c_int32 * MAX_OPS),
                ("round_each", ctypes.c_int32), ("has_bcast", ctypes.c_int32),
                ("bcast", Arr), ("bcast_dimensions", ctypes.c_int64 * MAX_RANK),
                ("bcast_data", ctypes.c_void_p), ("imm", ctypes.c_double * MAX_OPS)]


class Quant(ctypes.Structure):
    _fields_ = [("per_axis", ctypes.c_int32), ("quantization_dimension", ctypes.c_int32),
                ("n", ctypes.c_int64), ("scales", ctypes.POINTER(ctypes.c_float)),
                ("zero_points", ctypes.POINTER(ctypes.c_int32)),
                ("storage_min", ctypes.c_int32), ("storage_max", ctypes.c_int32)]


_lib_handle = None
_lib_lock = threading.Lock()


def lib():
    global _lib_handle
    with _lib_lock:
        if _lib_handle is None:
            h = ctypes.CDLL(build())
            P = ctypes.POINTER
            h.orc_linear_offset.argtypes = [P(Arr), P(ctypes.c_int64), P(ctypes.c_int64)]
            h.orc_broadcast_in_dim.argtypes = [P(Arr), ctypes.c_void_p, P(ctypes.c_int64), P(Arr), ctypes.c_void_p]
            h.orc_reduce.argtypes = [P(Arr), ctypes.c_void_p, P(Chain), P(ctypes.c_int64), ctypes.c_int,
                                     ctypes.c_int, ctypes.c_double, P(Arr), ctypes.c_void_p,
                                     P(ctypes.c_double)]
            h.orc_transpose.argtypes = [P(Arr), ctypes.c_void_p, P(Chain), P(ctypes.c_int64), ctypes.c_int,
                                        P(Chain), P(Arr), ctypes.c_void_p]
            h.orc_layout_convert.argtypes = [P(Arr), ctypes.c_void_p, P(ctypes.c_int64), ctypes.c_void_p]
            h.orc_reduce_max_argmax.argtypes = [P(Arr), ctypes.c_void_p, P(Arr), ctypes.c_void_p, P(ctypes.c_int64),
                                                ctypes.c_int, ctypes.c_double, ctypes.c_int64, P(Arr),
                                                ctypes.c_void_p, P(Arr), ctypes.c_void_p]
            h.orc_quant_fusion.argtypes = [P(Arr), ctypes.c_void_p, P(Quant), P(Chain), P(Arr),
                                           ctypes.c_void_p, P(Quant)]
            h.orc_quant_broadcast_in_dim.argtypes = [P(Arr), ctypes.c_void_p, P(Quant), P(ctypes.c_int64), P(Arr),
                                                     ctypes.c_void_p, P(ctypes.c_float), P(ctypes.c_int32),
                                                     P(ctypes.c_int32), P(ctypes.c_int64)]
            h.orc_quant_reshape.argtypes = [P(Arr), ctypes.c_void_p, P(Quant), P(Arr), ctypes.c_int32,
                                            ctypes.c_void_p]
            for name in ("orc_round_to", "orc_exp", "orc_log"):
                getattr(h, name).argtypes = [ctypes.c_double, ctypes.c_int]
                getattr(h, name).restype = ctypes.c_double
            h.orc_maximum.argtypes = [ctypes.c_double, ctypes.c_double]
            h.orc_maximum.restype = ctypes.c_double
            h.orc_quantize.argtypes = [P(Quant), ctypes.c_float, P(ctypes.c_int64)]
            h.orc_quantize.restype = ctypes.c_int
            h.orc_dequantize.argtypes = [P(Quant), ctypes.c_int32, P(ctypes.c_int64)]
            h.orc_dequantize.restype = ctypes.c_float
            h.orc_check_log_f32.argtypes = [ctypes.c_uint32, ctypes.c_int64, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_int64]
            h.orc_check_log_f32.restype = ctypes.c_int64
            h.orc_check_exp_f32.argtypes = [ctypes.c_uint32, ctypes.c_int64, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_int64]
            h.orc_check_exp_f32.restype = ctypes.c_int64
            h.orc_check_tanh_f32.argtypes = [ctypes.c_uint32, ctypes.c_int64, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_int64]
            h.orc_check_tanh_f32.restype = ctypes.c_int64
            h.orc_unresolved_count.restype = ctypes.c_int
            h.orc_set_num_threads.argtypes = [ctypes.c_int]
            h.orc_max_threads.restype = ctypes.c_int
            _lib_handle = h
    return _lib_handle


def default_m2m(rank: int):
    """Default layout: dimensions ordered major to minor, i.e. minor_to_major = [rank-1, ..., 0]."""
    return list(range(rank - 1, -1, -1))


def make_arr(dims, m2m, dtype) -> Arr:
    dims = list(dims)
    m2m = default_m2m(len(dims)) if m2m is None else list(m2m)
    if len(dims) > MAX_RANK or len(m2m) != len(dims):
        raise ValueError("bad rank / layout")
    a = Arr()
    a.rank = len(dims)
    a.dtype = DTYPES[dtype]
    for i, d in enumerate(dims):
        a.dims[i] = int(d)
    for i, d in enumerate(m2m):
        a.m2m[i] = int(d)
    return a


def _i64(values):
    values = list(values)
    return (ctypes.c_int64 * max(1, len(values)))(*[int(v) for v in values])


def _buf(data, dtype):
    arr = np.ascontiguousarray(data, dtype=NP_DTYPES[dtype])
    return arr, arr.ctypes.data_as(ctypes.c_void_p)


class _ChainKeep:
    """Holds a Chain and the numpy buffers it points into."""

    def __init__(self, spec):
        self.c = Chain()
        self.keep = []
        if spec is None:
            self.ptr = None
            return
        ops = list(spec.get("ops", []))
        if len(ops) > MAX_OPS:
            raise ValueError("too many ops")
        self.c.n_ops = len(ops)
        for i, op in enumerate(ops):
            if isinstance(op, (tuple, list)):  # (name, constant) for add_const / mul_const
                op, self.c.imm[i] = op[0], float(op[1])
            self.c.ops[i] = OPS[op]
        self.c.round_each = 1 if spec.get("round_each", True) else 0
        if "bcast" in spec and spec["bcast"] is not None:
            b = spec["bcast"]
            data, ptr = _buf(b["data"], b["dtype"])
            self.keep.append(data)
            self.c.has_bcast = 1
            self.c.bcast = make_arr(b["dims"], b.get("m2m"), b["dtype"])
            for i, d in enumerate(b["broadcast_dimensions"]):
                self.c.bcast_dimensions[i] = int(d)
            self.c.bcast_data = ptr
        self.ptr = ctypes.byref(self.c)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (code {rc})")


def linear_offset(dims, m2m, idx) -> int:
    a = make_arr(dims, m2m, "f32")
    out = ctypes.c_int64()
    _check(lib().orc_linear_offset(ctypes.byref(a), _i64(idx), ctypes.byref(out)), "linear_offset")
    return out.value


def broadcast_in_dim(data, dims, dtype, broadcast_dimensions, out_dims, m2m=None, out_m2m=None):
    a = make_arr(dims, m2m, dtype)
    o = make_arr(out_dims, out_m2m, dtype)
    src, sp = _buf(data, dtype)
    out = np.zeros(int(np.prod(out_dims)), dtype=NP_DTYPES[dtype])
    _check(lib().orc_broadcast_in_dim(ctypes.byref(a), sp, _i64(broadcast_dimensions), ctypes.byref(o),
                                      out.ctypes.data_as(ctypes.c_void_p)), "broadcast_in_dim")
    return out


def reduce(data, dims, dtype, dimensions, kind, init, out_dtype, m2m=None, out_m2m=None,
           prologue=None, want_abs_sum=False):
    """reduce over `dimensions`; returns the physical output buffer (and sum|term| if asked)."""
    a = make_arr(dims, m2m, dtype)
    red = set(int(d) for d in dimensions)
    out_dims = [d for i, d in enumerate(dims) if i not in red]
    o = make_arr(out_dims, out_m2m, out_dtype)
    src, sp = _buf(data, dtype)
    n_out = int(np.prod(out_dims)) if out_dims else 1
    out = np.zeros(n_out, dtype=NP_DTYPES[out_dtype])
    asum = np.zeros(n_out, dtype=np.float64)
    ch = _ChainKeep(prologue)
    rc = lib().orc_reduce(ctypes.byref(a), sp, ch.ptr, _i64(dimensions), len(list(dimensions)),
                          REDUCE_KINDS[kind], float(init), ctypes.byref(o),
                          out.ctypes.data_as(ctypes.c_void_p),
                          asum.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    _check(rc, "reduce")
    return (out, asum) if want_abs_sum else out


def transpose(data, dims, dtype, permutation, m2m=None, out_m2m=None, self_add=False,
              prologue=None, epilogue=None):
    a = make_arr(dims, m2m, dtype)
    out_dims = [dims[p] for p in permutation]
    o = make_arr(out_dims, out_m2m, dtype)
    src, sp = _buf(data, dtype)
    out = np.zeros(int(np.prod(out_dims)), dtype=NP_DTYPES[dtype])
    pro, epi = _ChainKeep(prologue), _ChainKeep(epilogue)
    rc = lib().orc_transpose(ctypes.byref(a), sp, pro.ptr, _i64(permutation), 1 if self_add else 0,
                             epi.ptr, ctypes.byref(o), out.ctypes.data_as(ctypes.c_void_p))
    _check(rc, "transpose")
    return out


def layout_convert(data, dims, dtype, m2m, out_m2m):
    a = make_arr(dims, m2m, dtype)
    src, sp = _buf(data, dtype)
    out = np.zeros(int(np.prod(dims)), dtype=NP_DTYPES[dtype])
    _check(lib().orc_layout_convert(ctypes.byref(a), sp, _i64(out_m2m), out.ctypes.data_as(ctypes.c_void_p)),
           "layout_convert")
    return out


class _QuantKeep:
    def __init__(self, spec):
        self.keep = []
        if spec is None:
            self.ptr = None
            return
        q = Quant()
        scales = np.ascontiguousarray(np.atleast_1d(spec["scales"]), dtype=np.float32)
        zps = np.ascontiguousarray(np.atleast_1d(spec["zero_points"]), dtype=np.int32)
        self.keep += [scales, zps]
        q.per_axis = 1 if spec.get("quantization_dimension") is not None else 0
        q.quantization_dimension = int(spec.get("quantization_dimension") or 0)
        q.n = len(scales)
        q.scales = scales.ctypes.data_as(ctypes.POINTER(ctypes.c_float))
        q.zero_points = zps.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        q.storage_min = int(spec.get("storage_min", -128))
        q.storage_max = int(spec.get("storage_max", 127))
        self.q = q
        self.ptr = ctypes.byref(q)


def quant_fusion(data, dims, in_dtype, in_q, out_m2m, out_dtype, out_q=None, m2m=None, float_ops=None):
    a = make_arr(dims, m2m, in_dtype)
    o = make_arr(dims, out_m2m, out_dtype)
    src, sp = _buf(data, in_dtype)
    out = np.zeros(int(np.prod(dims)), dtype=NP_DTYPES[out_dtype])
    qi, qo, ch = _QuantKeep(in_q), _QuantKeep(out_q), _ChainKeep(float_ops)
    rc = lib().orc_quant_fusion(ctypes.byref(a), sp, qi.ptr, ch.ptr, ctypes.byref(o),
                                out.ctypes.data_as(ctypes.c_void_p), qo.ptr)
    _check(rc, "quant_fusion")
    return out


def quant_broadcast_in_dim(data, dims, q, broadcast_dimensions, out_dims, m2m=None, out_m2m=None, dtype="s8"):
    """broadcast_in_dim of a quantized tensor: returns (codes in the result layout, result parameters
    {"scales", "zero_points", "quantization_dimension"})."""
    a, o = make_arr(dims, m2m, dtype), make_arr(out_dims, out_m2m, dtype)
    src, sp = _buf(data, dtype)
    out = np.zeros(max(1, int(np.prod(out_dims))), dtype=NP_DTYPES[dtype])
    cap = max([1] + [int(d) for d in out_dims])
    rs = np.zeros(cap, np.float32)
    rz = np.zeros(cap, np.int32)
    rqd, rn = ctypes.c_int32(), ctypes.c_int64()
    qk = _QuantKeep(q)
    rc = lib().orc_quant_broadcast_in_dim(ctypes.byref(a), sp, qk.ptr, _i64(broadcast_dimensions), ctypes.byref(o),
                                          out.ctypes.data_as(ctypes.c_void_p),
                                          rs.ctypes.data_as(ctypes.POINTER(ctypes.c_float)),
                                          rz.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), ctypes.byref(rqd),
                                          ctypes.byref(rn))
    _check(rc, "quant_broadcast_in_dim")
    params = {"scales": rs[:rn.value].copy(), "zero_points": rz[:rn.value].copy(),
              "quantization_dimension": None if rqd.value < 0 else rqd.value}
    return out[:int(np.prod(out_dims))], params


def reshape(data, dims, out_dims, dtype, m2m=None, out_m2m=None, q=None, result_qdim=-1):
    """reshape (lexicographic order kept); q: the operand's quantization (None for plain arrays) and
    result_qdim the result type's quantization dimension (-1 per-tensor)."""
    a, o = make_arr(dims, m2m, dtype), make_arr(out_dims, out_m2m, dtype)
    src, sp = _buf(data, dtype)
    out = np.zeros(max(1, int(np.prod(out_dims))), dtype=NP_DTYPES[dtype])
    qk = _QuantKeep(q)
    rc = lib().orc_quant_reshape(ctypes.byref(a), sp, qk.ptr, ctypes.byref(o), int(result_qdim),
                                 out.ctypes.data_as(ctypes.c_void_p))
    _check(rc, "reshape")
    return out[:int(np.prod(out_dims))]


QUANT_BINARY_OPS = {"add": 0, "divide": 1, "maximum": 2, "minimum": 3, "multiply": 4}


def quant_binary(op, lhs, rhs, dims, lhs_q, rhs_q, out_q, lhs_m2m=None, rhs_m2m=None, out_m2m=None):
    """quantize(op(dequantize(lhs), dequantize(rhs))) with per-tensor s8 operands."""
    a, b, o = make_arr(dims, lhs_m2m, "s8"), make_arr(dims, rhs_m2m, "s8"), make_arr(dims, out_m2m, "s8")
    lb, lp = _buf(lhs, "s8")
    rb, rp = _buf(rhs, "s8")
    out = np.zeros(max(1, int(np.prod(dims))), dtype=np.int8)
    ql, qr, qo = _QuantKeep(lhs_q), _QuantKeep(rhs_q), _QuantKeep(out_q)
    rc = lib().orc_quant_binary(QUANT_BINARY_OPS[op], ctypes.byref(a), lp, ql.ptr, ctypes.byref(b), rp, qr.ptr,
                                ctypes.byref(o), out.ctypes.data_as(ctypes.c_void_p), qo.ptr)
    _check(rc, "quant_binary")
    return out[:int(np.prod(dims))]


def quantize(spec, real, idx=()):
    q = _QuantKeep(spec)
    return lib().orc_quantize(q.ptr, float(real), _i64(idx or [0]))


def dequantize(spec, code, idx=()):
    q = _QuantKeep(spec)
    return lib().orc_dequantize(q.ptr, int(code), _i64(idx or [0]))


def reduce_max_argmax(data, dims, dtype, dimensions, init_value, init_index, m2m=None, out_m2m=None,
                      indices=None, idx_m2m=None, out_idx_m2m=None):
    """Variadic max/argmax reduce: returns (values, indices); indices None means the position along
    the single reduced dimension."""
    a = make_arr(dims, m2m, dtype)
    kept = [d for d in range(len(dims)) if d not in dimensions]
    out_dims = [dims[d] for d in kept]
    o = make_arr(out_dims, out_m2m, dtype)
    oi = make_arr(out_dims, out_idx_m2m, "s32")
    src, sp = _buf(data, dtype)
    if indices is not None:
        ka = make_arr(dims, idx_m2m if idx_m2m is not None else m2m, "s32")
        kbuf, kp = _buf(indices, "s32")
    else:
        ka, kbuf, kp = make_arr(dims, m2m, "s32"), None, None
    vals = np.zeros(max(1, int(np.prod(out_dims))), dtype=NP_DTYPES[dtype])
    idx = np.zeros(max(1, int(np.prod(out_dims))), dtype=np.int32)
    rc = lib().orc_reduce_max_argmax(ctypes.byref(a), sp, ctypes.byref(ka), kp, _i64(dimensions), len(dimensions),
                                     ctypes.c_double(init_value), ctypes.c_int64(init_index), ctypes.byref(o),
                                     vals.ctypes.data_as(ctypes.c_void_p), ctypes.byref(oi),
                                     idx.ctypes.data_as(ctypes.c_void_p))
    _check(rc, "reduce_max_argmax")
    n = int(np.prod(out_dims))
    return vals[:n], idx[:n]


def round_to(x, dtype):
    return lib().orc_round_to(float(x), DTYPES[dtype])


def exp(x, dtype):
    return lib().orc_exp(float(x), DTYPES[dtype])


def log(x, dtype):
    return lib().orc_log(float(x), DTYPES[dtype])


def maximum(a, b):
    return lib().orc_maximum(float(a), float(b))


def check_log_f32(first_bits: int, cand_bits: np.ndarray, max_report: int = 16):
    """Count mismatches between cand_bits (uint32 patterns of f32 log results for consecutive inputs
    starting at first_bits) and the oracle's correctly rounded log. Returns (count, examples)."""
    cand = np.ascontiguousarray(cand_bits, dtype=np.uint32)
    report = np.zeros(max_report, dtype=np.uint32)
    bad = lib().orc_check_log_f32(first_bits, cand.size, cand.ctypes.data, report.ctypes.data, max_report)
    return int(bad), report[: min(bad, max_report)].tolist()


def check_exp_f32(first_bits: int, cand_bits: np.ndarray, max_report: int = 16):
    """Count mismatches between cand_bits (uint32 patterns of f32 exp results for consecutive inputs
    starting at first_bits) and the oracle's correctly rounded exp. Returns (count, examples)."""
    cand = np.ascontiguousarray(cand_bits, dtype=np.uint32)
    report = np.zeros(max_report, dtype=np.uint32)
    bad = lib().orc_check_exp_f32(first_bits, cand.size, cand.ctypes.data, report.ctypes.data, max_report)
    return int(bad), report[: min(bad, max_report)].tolist()


def check_tanh_f32(first_bits: int, cand_bits: np.ndarray, max_report: int = 16):
    """Count mismatches between cand_bits (uint32 patterns of f32 tanh results for consecutive inputs
    starting at first_bits) and the oracle's correctly rounded tanh. Returns (count, examples)."""
    cand = np.ascontiguousarray(cand_bits, dtype=np.uint32)
    report = np.zeros(max_report, dtype=np.uint32)
    bad = lib().orc_check_tanh_f32(first_bits, cand.size, cand.ctypes.data, report.ctypes.data, max_report)
    return int(bad), report[: min(bad, max_report)].tolist()


def unresolved_count() -> int:
    """Elements whose rounding could not be decided even in long double (expected 0)."""
    return lib().orc_unresolved_count()


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


def max_threads() -> int:
    return lib().orc_max_threads()
