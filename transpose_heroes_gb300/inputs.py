"""Seeded synthetic inputs for the five hero fusions (and scaled-down variants).

This module holds only data generation: random draws, the packing of draws into 16-bit float bit
patterns, and plain descriptions of each fusion (shapes, layouts, element types, parameters). It
contains none of the fused computation. Both the CUDA path and the CPU oracle receive the arrays it
returns, so the two always see identical bytes.

Every buffer is produced in PHYSICAL order: i.i.d. draws fill memory in address order, which is the
same distribution whatever the layout. Draws use numpy's PCG64 generator; U(a, b) draws are numpy's
half-open [a, b); integer draws are inclusive of both ends.

The full-size workloads follow the five fusions named for this path:
  row_reduce_exp      x f32[256,512]{1,0} ~ U(-1,1); out f32[256] = reduce-add over dim 1 of exp(x)
  transpose_log       p f32[8192,8192]{1,0} ~ U(0.5,2); out = log(p) + transpose(log(p), {1,0})
  col_reduce_max      x bf16[8192,16384]{1,0} ~ N(0,1); out bf16[16384] = reduce-max over dim 0
  bcast_exp_reduce    x bf16[8,1,1280,16384]{3,2,0,1} ~ N(0,1), b bf16[16384] ~ U(-1,1) on dim 3;
                      out f32[8,1,1280] = reduce-add over dim 3 of add(exp(x), b)
  quant_relayout      q s8[4096,4096]{1,0} ~ U[-128,127], per-axis (dim 1) scale ~ U(0.001,0.1),
                      zero_point ~ U[-20,20]; dequantize, relayout {1,0} -> {0,1}, quantize per-tensor
                      scale 0.05, zero_point 0, storage [-128,127]
"""

from __future__ import annotations

import dataclasses
from typing import Any, Optional

import numpy as np

ELEM_BYTES = {"f32": 4, "bf16": 2, "f16": 2, "f64": 8, "s8": 1, "u8": 1, "s32": 4}


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Pack f32 draws into bf16 bit patterns, rounding to nearest with ties to even (finite input)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to f32 (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def uniform_f32(g: np.random.Generator, n: int, lo: float, hi: float) -> np.ndarray:
    return g.uniform(lo, hi, size=n).astype(np.float32)


def normal_bf16(g: np.random.Generator, n: int) -> np.ndarray:
    return f32_to_bf16_bits(g.standard_normal(size=n, dtype=np.float32))


def uniform_bf16(g: np.random.Generator, n: int, lo: float, hi: float) -> np.ndarray:
    return f32_to_bf16_bits(uniform_f32(g, n, lo, hi))


def integers(g: np.random.Generator, n: int, lo: int, hi: int, dtype) -> np.ndarray:
    return g.integers(lo, hi, size=n, endpoint=True).astype(dtype)


@dataclasses.dataclass
class Fusion:
    """Plain description of one fusion instance and its input buffers (physical order)."""

    name: str
    kind: str                      # "reduce" | "transpose" | "quant" | "argmax"
    dims: list
    m2m: list
    dtype: str
    data: np.ndarray
    # reduce
    dimensions: Optional[list] = None
    reduce_kind: Optional[str] = None
    init: float = 0.0
    # transpose
    permutation: Optional[list] = None
    self_add: bool = False
    # quant
    in_q: Optional[dict] = None
    out_q: Optional[dict] = None
    # quantized binary op: the op name and the second operand (physical order)
    op: Optional[str] = None
    rhs: Optional[np.ndarray] = None
    # common
    prologue: Optional[dict] = None
    epilogue: Optional[dict] = None
    out_dims: Optional[list] = None
    out_m2m: Optional[list] = None
    out_dtype: Optional[str] = None
    description: str = ""

    @property
    def elements(self) -> int:
        """Logical elements of the hero's input (for transposes this equals output elements)."""
        return int(np.prod(self.dims))

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes a single pass must move: every input element read once, every output written once,
        side operands (broadcast vector, quantization parameters) counted once."""
        b = self.elements * ELEM_BYTES[self.dtype]
        b += int(np.prod(self.out_dims)) * ELEM_BYTES[self.out_dtype] if self.out_dims else ELEM_BYTES[self.out_dtype]
        for chain in (self.prologue, self.epilogue):
            if chain and chain.get("bcast") is not None:
                bc = chain["bcast"]
                b += int(np.prod(bc["dims"])) * ELEM_BYTES[bc["dtype"]]
        if self.in_q is not None:
            # scales f32 + zero points stored in the storage type
            b += len(np.atleast_1d(self.in_q["scales"])) * (4 + ELEM_BYTES[self.dtype])
        if self.kind == "argmax":  # the s32 index output beside the values
            b += int(np.prod(self.out_dims)) * 4
        if self.kind == "quant_binary":  # the second operand
            b += self.elements * ELEM_BYTES[self.dtype]
        return int(b)


def _default_m2m(rank):
    return list(range(rank - 1, -1, -1))


def row_reduce_exp(seed: int = 1, rows: int = 256, cols: int = 512) -> Fusion:
    g = rng(seed)
    return Fusion(
        name=f"row_reduce_exp_f32_{rows}x{cols}", kind="reduce", dims=[rows, cols], m2m=[1, 0], dtype="f32",
        data=uniform_f32(g, rows * cols, -1.0, 1.0), dimensions=[1], reduce_kind="add", init=0.0,
        prologue={"ops": ["exp"], "round_each": True},
        out_dims=[rows], out_m2m=[0], out_dtype="f32",
        description="out f32[rows] = reduce-add over dim 1 of exp(x), x f32[rows,cols]{1,0} ~ U(-1,1), init 0")


def transpose_log(seed: int = 1, n: int = 8192) -> Fusion:
    g = rng(seed)
    return Fusion(
        name=f"transpose_selfadd_log_f32_{n}x{n}", kind="transpose", dims=[n, n], m2m=[1, 0], dtype="f32",
        data=uniform_f32(g, n * n, 0.5, 2.0), permutation=[1, 0], self_add=True,
        prologue={"ops": ["log"], "round_each": True},
        out_dims=[n, n], out_m2m=[1, 0], out_dtype="f32",
        description="out = add(log(p), transpose(log(p), {1,0})), p f32[n,n]{1,0} ~ U(0.5,2)")


def col_reduce_max(seed: int = 1, rows: int = 8192, cols: int = 16384) -> Fusion:
    g = rng(seed)
    return Fusion(
        name=f"col_reduce_max_bf16_{rows}x{cols}", kind="reduce", dims=[rows, cols], m2m=[1, 0], dtype="bf16",
        data=normal_bf16(g, rows * cols), dimensions=[0], reduce_kind="max", init=float("-inf"),
        prologue=None, out_dims=[cols], out_m2m=[0], out_dtype="bf16",
        description="out bf16[cols] = reduce-max over dim 0 of x, x bf16[rows,cols]{1,0} ~ N(0,1), init -inf, f32 accumulation")


def bcast_exp_reduce(seed: int = 1, d0: int = 8, d2: int = 1280, d3: int = 16384) -> Fusion:
    g = rng(seed)
    x = normal_bf16(g, d0 * d2 * d3)
    b = uniform_bf16(g, d3, -1.0, 1.0)
    return Fusion(
        name=f"bcast_exp_row_reduce_bf16_{d0}x1x{d2}x{d3}", kind="reduce", dims=[d0, 1, d2, d3],
        m2m=[3, 2, 0, 1], dtype="bf16", data=x, dimensions=[3], reduce_kind="add", init=0.0,
        prologue={"ops": ["exp", "add_bcast"], "round_each": True,
                  "bcast": {"data": b, "dims": [d3], "m2m": [0], "dtype": "bf16", "broadcast_dimensions": [3]}},
        out_dims=[d0, 1, d2], out_m2m=[2, 1, 0], out_dtype="f32",
        description="out f32[d0,1,d2] = reduce-add over dim 3 of add(exp(x), broadcast(b, {3})), "
                    "x bf16[d0,1,d2,d3]{3,2,0,1} ~ N(0,1), b bf16[d3] ~ U(-1,1)")


def quant_relayout(seed: int = 1, n0: int = 4096, n1: int = 4096) -> Fusion:
    g = rng(seed)
    q = integers(g, n0 * n1, -128, 127, np.int8)
    scales = uniform_f32(g, n1, 0.001, 0.1)
    zps = integers(g, n1, -20, 20, np.int32)
    return Fusion(
        name=f"quant_relayout_s8_{n0}x{n1}", kind="quant", dims=[n0, n1], m2m=[1, 0], dtype="s8", data=q,
        in_q={"scales": scales, "zero_points": zps, "quantization_dimension": 1,
              "storage_min": -128, "storage_max": 127},
        out_q={"scales": np.array([0.05], dtype=np.float32), "zero_points": np.array([0], dtype=np.int32),
               "quantization_dimension": None, "storage_min": -128, "storage_max": 127},
        out_dims=[n0, n1], out_m2m=[0, 1], out_dtype="s8",
        description="per-axis (dim 1) dequantize of q s8[n0,n1]{1,0}, relayout to {0,1}, quantize per-tensor 0.05:0")


# The loop fusion of "XLA:GPU Emitters", section "Loop emitter" (the GELU function and its HLO module
# in "Reproducer"): bf16 multiply/add/tanh with the HLO's constants, every op rounded to bf16, as one
# chain that folds the parameter into a running value.
GELU_CHAIN = [
    "mul_input",                # square = x * x
    "mul_input",                # cube = square * x
    ("mul_const", 0.044708),    # * constant(0.044708)
    "add_input",                # x + ...
    ("mul_const", 0.79785),     # * constant(0.79785)
    "tanh",
    ("add_const", 1.0),         # + constant(1)
    ("mul_const", 0.5),         # * constant(0.5)
    "mul_input",                # x * ...
]


def gelu_bf16(seed: int = 1, dims=(6, 512, 4096), data=None) -> Fusion:
    """x bf16[6,512,4096]{2,1,0} ~ N(0,1) (activations; the pages give no distribution), out bf16 same
    shape and layout = gelu(x) with the per-op bf16 rounding of the HLO."""
    dims = list(dims)
    n = int(np.prod(dims))
    if data is None:
        data = normal_bf16(rng(seed), n)
    m2m = _default_m2m(len(dims))
    return Fusion(
        name="gelu_bf16_" + "x".join(str(d) for d in dims), kind="transpose", dims=dims, m2m=m2m, dtype="bf16",
        data=data, permutation=list(range(len(dims))), self_add=False,
        prologue={"ops": list(GELU_CHAIN), "round_each": True}, out_dims=dims, out_m2m=m2m, out_dtype="bf16",
        description="loop fusion: gelu(x) (tanh form) on x bf16[6,512,4096] ~ N(0,1), bf16 per op")


def argmax_f32(seed: int = 1, rows: int = 4096, cols: int = 32768) -> Fusion:
    """Variadic max/argmax reduce (XLA Operation Semantics, "Variadic Reduce") over the last dim of
    f32[rows, cols]{1,0} ~ N(0,1) with the position as index (a logits-like row argmax; the pages give
    no size); out f32[rows] values and s32[rows] indices."""
    g = rng(seed)
    return Fusion(
        name=f"argmax_f32_{rows}x{cols}", kind="argmax", dims=[rows, cols], m2m=[1, 0], dtype="f32",
        data=g.standard_normal(rows * cols, dtype=np.float32), dimensions=[1], reduce_kind="max_argmax",
        init=float("-inf"), out_dims=[rows], out_m2m=[0], out_dtype="f32",
        description=f"max/argmax over dim 1 of x f32[{rows},{cols}]{{1,0}} ~ N(0,1), index = position")


def quant_add_s8(seed: int = 1, n0: int = 4096, n1: int = 4096) -> Fusion:
    """Quantized add (StableHLO Specification, "add" on quantized types; the quantized test case of
    "StableHLO Quantization" adds two i8:f32 0.3 tensors): lhs, rhs s8[n0,n1]{1,0} ~ U[-128,127],
    both per-tensor 0.3:0, result per-tensor 0.3:0. `data` holds lhs, `rhs` the second operand."""
    g = rng(seed)
    n = n0 * n1
    f = Fusion(
        name=f"quant_add_s8_{n0}x{n1}", kind="quant_binary", dims=[n0, n1], m2m=[1, 0], dtype="s8",
        data=integers(g, n, -128, 127, np.int8),
        in_q={"scales": np.float32([0.3]), "zero_points": np.int32([0]), "quantization_dimension": None},
        out_q={"scales": np.float32([0.3]), "zero_points": np.int32([0]), "quantization_dimension": None,
               "storage_min": -128, "storage_max": 127},
        out_dims=[n0, n1], out_m2m=[1, 0], out_dtype="s8",
        description=f"quantized add of s8[{n0},{n1}] i8:f32 0.3 operands, result i8:f32 0.3",
        op="add")
    f.rhs = integers(g, n, -128, 127, np.int8)
    return f


def transpose3_exp_abs(seed: int = 1, dims=(512, 640, 680)) -> Fusion:
    """The transpose fusion of "XLA:GPU Emitters", section "Transpose emitter" (exp -> transpose with
    permutation {2,1,0} -> abs, printed on f32[20,160,170]), scaled up so that it streams HBM: x
    f32[d0,d1,d2]{2,1,0} ~ U(-3,3) (the pages give no distribution), out f32[d2,d1,d0]{2,1,0}."""
    dims = list(dims)
    n = int(np.prod(dims))
    out_dims = [dims[2], dims[1], dims[0]]
    return Fusion(
        name="transpose3_exp_abs_f32_" + "x".join(str(d) for d in dims), kind="transpose", dims=dims,
        m2m=[2, 1, 0], dtype="f32", data=uniform_f32(rng(seed), n, -3.0, 3.0), permutation=[2, 1, 0],
        self_add=False, prologue={"ops": ["exp"], "round_each": True}, epilogue={"ops": ["abs"], "round_each": True},
        out_dims=out_dims, out_m2m=[2, 1, 0], out_dtype="f32",
        description=f"abs(transpose(exp(x), {{2,1,0}})), x f32[{dims[0]},{dims[1]},{dims[2]}]{{2,1,0}} ~ U(-3,3)")


def sum_exp_f32(seed: int = 1, n: int = 1 << 26) -> Fusion:
    """A whole array reduced to one value: sum of exp(x) over x f32[n] ~ U(-1,1), seen as [1, n] (the
    row reduce with a single row, which splits the row across blocks)."""
    g = rng(seed)
    return Fusion(
        name=f"sum_exp_f32_{n}", kind="reduce", dims=[1, n], m2m=[1, 0], dtype="f32",
        data=uniform_f32(g, n, -1.0, 1.0), dimensions=[1], reduce_kind="add", init=0.0,
        prologue={"ops": ["exp"], "round_each": True}, out_dims=[1], out_m2m=[0], out_dtype="f32",
        description=f"out f32[1] = reduce-add over dim 1 of exp(x), x f32[1,{n}] ~ U(-1,1)")


# The five full-size workloads, in a fixed order.
FULL = {
    "row_reduce_exp": row_reduce_exp,
    "transpose_log": transpose_log,
    "col_reduce_max": col_reduce_max,
    "bcast_exp_reduce": bcast_exp_reduce,
    "quant_relayout": quant_relayout,
}

# Scaled-down shapes that still span several tiles and end in ragged tails.
SMALL = {
    "row_reduce_exp": dict(rows=37, cols=1000),
    "transpose_log": dict(n=333),
    "col_reduce_max": dict(rows=301, cols=1030),
    "bcast_exp_reduce": dict(d0=3, d2=45, d3=2003),
    "quant_relayout": dict(n0=301, n1=517),
}


def full(name: str, seed: int = 1) -> Fusion:
    return FULL[name](seed=seed)


def small(name: str, seed: int = 1, **overrides: Any) -> Fusion:
    kw = dict(SMALL[name])
    kw.update(overrides)
    return FULL[name](seed=seed, **kw)
