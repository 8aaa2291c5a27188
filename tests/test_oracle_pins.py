"""Pins for the CPU oracle: the pages' worked examples, closed forms, invariants, exact arithmetic
(Python's decimal / fractions) and brute force against numpy on tiny inputs.

These run without a GPU. Each check is chosen so that a plausible slip in the oracle -- a wrong
stride order, a transposed operand, a dropped rounding, ties away from zero instead of to even,
the wrong quantization axis -- fails at least one of them.
"""

import itertools
import math
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

from conftest import load_golden

getcontext().prec = 80


# ---------------------------------------------------------------------------------------------
# helpers (test-side, independent of the oracle): logical <-> physical buffers via numpy
# ---------------------------------------------------------------------------------------------
def to_physical(arr, m2m):
    order = list(reversed(m2m))  # major -> minor
    return np.ascontiguousarray(np.transpose(arr, order)).ravel()


def from_physical(buf, dims, m2m):
    order = list(reversed(m2m))
    phys = np.asarray(buf).reshape([dims[d] for d in order])
    return np.transpose(phys, np.argsort(order))


def all_layouts(rank):
    return [list(p) for p in itertools.permutations(range(rank))]


def f32_neighbors(y):
    y = np.float32(y)
    return np.nextafter(y, np.float32(-np.inf)), np.nextafter(y, np.float32(np.inf))


def exact_between_midpoints(exact: Decimal, y: float, lo: float, hi: float) -> bool:
    """True if `exact` lies strictly inside the rounding interval of y (between the midpoints to its
    neighbours lo and hi); midpoints are computed exactly in Decimal."""
    y, lo, hi = Decimal(float(y)), Decimal(float(lo)), Decimal(float(hi))
    return (y + lo) / 2 < exact < (y + hi) / 2


# ---------------------------------------------------------------------------------------------
# layout addressing (XLA Shapes and Layout, "Layout")
# ---------------------------------------------------------------------------------------------
def test_layout_2x3_memory_orders(orc):
    g = load_golden("layout_2x3.txt")
    letters = g["logical"][0] + g["logical"][1]
    logical = np.arange(6, dtype=np.int8)  # a..f in row order: a=0 ... f=5
    for key, memory in g["memory"].items():
        m2m = [int(v) for v in key.split(",")]
        # offsets of each logical element
        mem = [None] * 6
        for i in range(2):
            for j in range(3):
                mem[orc.linear_offset(g["dims"], m2m, [i, j])] = g["logical"][i][j]
        assert mem == memory
        # and the same through a layout conversion of the row-major buffer
        out = orc.layout_convert(logical, g["dims"], "s8", [1, 0], m2m)
        assert [letters[v] for v in out] == memory


def test_default_layout_is_major_to_minor(orc):
    g = load_golden("layout_2x3.txt")
    assert orc.default_m2m(3) == g["default_m2m_rank3"]


@pytest.mark.parametrize("dims", [[3, 4, 5], [2, 1, 3, 2], [5, 7]])
def test_linear_offset_matches_numpy_strides(orc, dims):
    for m2m in all_layouts(len(dims)):
        order = list(reversed(m2m))
        phys_shape = [dims[d] for d in order]
        for idx in itertools.product(*[range(d) for d in dims]):
            want = np.ravel_multi_index(tuple(idx[d] for d in order), phys_shape)
            assert orc.linear_offset(dims, m2m, idx) == want


def test_layout_convert_roundtrip_and_numpy(orc):
    g = np.random.default_rng(5)
    dims = [3, 5, 4]
    logical = g.integers(-100, 100, size=dims).astype(np.int8)
    for a in all_layouts(3):
        buf_a = to_physical(logical, a)
        for b in all_layouts(3):
            out = orc.layout_convert(buf_a, dims, "s8", a, b)
            assert np.array_equal(out, to_physical(logical, b))
            back = orc.layout_convert(out, dims, "s8", b, a)
            assert np.array_equal(back, buf_a)


def test_layout_convert_sizes_zero_and_one(orc):
    assert orc.layout_convert(np.zeros(0, np.float32), [0, 3], "f32", [1, 0], [0, 1]).size == 0
    x = np.arange(5, dtype=np.float32)
    assert np.array_equal(orc.layout_convert(x, [1, 5], "f32", [1, 0], [0, 1]), x)


# ---------------------------------------------------------------------------------------------
# transpose (XLA:GPU Emitters, "Indexing transformations" / "Transpose emitter")
# ---------------------------------------------------------------------------------------------
def test_transpose_map_20x40(orc):
    g = load_golden("transpose_maps.txt")["map_2d"]
    x = np.arange(20 * 40, dtype=np.float32)  # in[d1', d0'] = 40*d1' + d0'
    out = orc.transpose(x, g["in_dims"], "f32", g["permutation"]).reshape(g["out_dims"])
    for d0 in range(40):
        for d1 in range(20):
            assert out[d0, d1] == x[d1 * 40 + d0]  # output (d0, d1) reads input (d1, d0)


def test_transpose_emitter_example_exp_abs(orc):
    g = load_golden("transpose_maps.txt")["emitter_3d"]
    rng = np.random.default_rng(3)
    dims = g["in_dims"]
    x = rng.uniform(-3, 3, size=int(np.prod(dims))).astype(np.float32)
    out = orc.transpose(x, dims, "f32", g["permutation"], prologue={"ops": ["exp"]},
                        epilogue={"ops": ["abs"]}).reshape(g["out_dims"])
    xl = x.reshape(dims)
    # exact exp rounded to f32 checked on a sample through Decimal
    for (i, j, k) in [(0, 0, 0), (19, 159, 169), (7, 80, 3), (11, 2, 150)]:
        v = float(xl[i, j, k])
        y = float(out[k, j, i])
        lo, hi = f32_neighbors(y)
        assert exact_between_midpoints(Decimal(v).exp(), y, lo, hi)
    # the whole mapping: out[k, j, i] == |f32(exp(x[i, j, k]))| within 1 ulp of numpy's exp
    ref = np.abs(np.exp(xl.astype(np.float64)).astype(np.float32)).transpose(2, 1, 0)
    assert np.array_equal(out.shape, ref.shape)
    assert np.max(np.abs(out.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))) <= 1


@pytest.mark.parametrize("rank", [1, 2, 3, 4])
def test_transpose_all_permutations_vs_numpy(orc, rank):
    rng = np.random.default_rng(rank)
    dims = [2, 3, 4, 5][:rank]
    logical = rng.integers(-1000, 1000, size=dims).astype(np.float32)
    layouts = all_layouts(rank)
    for perm in itertools.permutations(range(rank)):
        out_dims = [dims[p] for p in perm]
        in_m2m = layouts[(sum(perm) + 1) % len(layouts)]
        out_m2m = layouts[(perm[0] + 2) % len(layouts)]
        buf = to_physical(logical, in_m2m)
        out = orc.transpose(buf, dims, "f32", list(perm), m2m=in_m2m, out_m2m=out_m2m,
                            prologue={"ops": ["neg"]})
        want = -np.transpose(logical, perm)
        assert np.array_equal(from_physical(out, out_dims, out_m2m), want)


def test_transpose_moves_integers_exactly(orc):
    """A transpose is a pure index map: 32-bit integers keep all their bits (no float rounding)."""
    rng = np.random.default_rng(19)
    dims = [3, 5, 7]
    logical = rng.integers(-2 ** 31, 2 ** 31 - 1, size=dims).astype(np.int32)
    for perm in itertools.permutations(range(3)):
        out = orc.transpose(logical.ravel(), dims, "s32", list(perm))
        assert np.array_equal(out.reshape([dims[p] for p in perm]), np.transpose(logical, perm))


def test_transpose_self_add(orc):
    rng = np.random.default_rng(7)
    n = 9
    x = rng.uniform(-5, 5, size=(n, n)).astype(np.float32)
    out = orc.transpose(x.ravel(), [n, n], "f32", [1, 0], self_add=True,
                        prologue={"ops": ["abs"]}).reshape(n, n)
    want = (np.abs(x).astype(np.float64) + np.abs(x).T.astype(np.float64)).astype(np.float32)
    assert np.array_equal(out, want)


def test_transpose_self_add_log_symmetric_and_correct(orc):
    rng = np.random.default_rng(11)
    n = 17
    p = rng.uniform(0.5, 2.0, size=n * n).astype(np.float32)
    out = orc.transpose(p, [n, n], "f32", [1, 0], self_add=True, prologue={"ops": ["log"]}).reshape(n, n)
    assert np.array_equal(out.view(np.uint32), out.T.view(np.uint32))  # bitwise symmetric
    P = p.reshape(n, n)
    for i, j in [(0, 0), (3, 5), (16, 2)]:
        li, lj = orc.log(P[i, j], "f32"), orc.log(P[j, i], "f32")
        assert out[i, j] == np.float32(np.float64(li) + np.float64(lj))


# ---------------------------------------------------------------------------------------------
# reduce (StableHLO Specification "reduce"; XLA Operation Semantics "Reduce")
# ---------------------------------------------------------------------------------------------
def test_reduce_spec_example(orc):
    g = load_golden("reduce_examples.txt")["spec"]
    x = np.array(g["input"], dtype=np.float32).ravel()
    out = orc.reduce(x, [1, 6], "f32", g["dimensions"], "add", g["init"], "f32")
    assert out.tolist() == g["result"]


@pytest.mark.parametrize("m2m", all_layouts(3))
def test_reduce_xla_3d_examples(orc, m2m):
    g = load_golden("reduce_examples.txt")["xla_3d"]
    logical = np.array([g["slab"]] * g["replicas"], dtype=np.float32)  # [4, 2, 3]
    buf = to_physical(logical, m2m)
    for case in g["cases"]:
        out = orc.reduce(buf, [4, 2, 3], "f32", case["dimensions"], "add", 0.0, "f32", m2m=m2m)
        want = np.array(case["result"], dtype=np.float32).ravel()
        assert np.array_equal(out, want), (case, m2m)


def test_reduce_closed_forms(orc):
    n = 1000
    iota = np.arange(n, dtype=np.float32)
    assert orc.reduce(iota, [n], "f32", [0], "add", 0.0, "f32")[0] == n * (n - 1) / 2
    assert orc.reduce(iota, [n], "f32", [0], "max", -np.inf, "f32")[0] == n - 1
    assert orc.reduce(np.ones(n, np.float32), [n], "f32", [0], "add", 3.0, "f32")[0] == n + 3  # init once
    # empty reduced dimension: the init value
    assert orc.reduce(np.zeros(0, np.float32), [0], "f32", [0], "add", 2.5, "f32")[0] == 2.5
    assert orc.reduce(np.zeros(0, np.float32), [4, 0], "f32", [1], "max", -np.inf, "f32").tolist() == [-np.inf] * 4


@pytest.mark.parametrize("kind", ["add", "max"])
def test_reduce_brute_force_vs_numpy(orc, kind):
    rng = np.random.default_rng(13)
    dims = [3, 4, 5]
    logical = rng.standard_normal(dims).astype(np.float32)
    for m2m in all_layouts(3):
        buf = to_physical(logical, m2m)
        for r in range(1, 4):
            for red in itertools.combinations(range(3), r):
                kept = [d for d in range(3) if d not in red]
                out_m2m = orc.default_m2m(len(kept))
                init = 0.0 if kind == "add" else -np.inf
                out = orc.reduce(buf, dims, "f32", list(red), kind, init, "f64", m2m=m2m)
                if kind == "add":
                    want = logical.astype(np.float64).sum(axis=red)
                    assert np.allclose(out, np.ravel(want), rtol=1e-15, atol=1e-15)
                else:
                    want = logical.max(axis=red).astype(np.float64)
                    assert np.array_equal(out, np.ravel(want))
                del out_m2m


def test_reduce_output_layout(orc):
    rng = np.random.default_rng(17)
    dims = [4, 6, 5]
    logical = rng.integers(-9, 9, size=dims).astype(np.float32)
    want = logical.sum(axis=1)  # [4, 5]
    for out_m2m in ([1, 0], [0, 1]):
        out = orc.reduce(logical.ravel(), dims, "f32", [1], "add", 0.0, "f32", out_m2m=out_m2m)
        assert np.array_equal(from_physical(out, [4, 5], out_m2m), want)


def test_maximum_semantics(orc):
    g = load_golden("elementwise_examples.txt")["maximum"]
    for a, b, c in zip(np.ravel(g["lhs"]), np.ravel(g["rhs"]), np.ravel(g["result"])):
        assert orc.maximum(a, b) == c
    assert math.isnan(orc.maximum(float("nan"), 1.0)) and math.isnan(orc.maximum(1.0, float("nan")))
    assert math.copysign(1.0, orc.maximum(-0.0, 0.0)) == 1.0
    assert math.copysign(1.0, orc.maximum(0.0, -0.0)) == 1.0
    # a NaN anywhere in a reduced column propagates
    x = np.array([1.0, np.nan, 3.0, 2.0], dtype=np.float32)
    assert math.isnan(orc.reduce(x, [4], "f32", [0], "max", -np.inf, "f32")[0])
    x = np.array([-0.0, 0.0, -0.0], dtype=np.float32)
    r = orc.reduce(x, [3], "f32", [0], "max", -np.inf, "f32")[0]
    assert r == 0 and not np.signbit(r)


def test_max_reduce_to_bf16_is_exact_member(orc):
    import transpose_heroes_gb300.inputs as inp

    rng = inp.rng(2)
    x = inp.normal_bf16(rng, 64 * 33)
    out = orc.reduce(x, [64, 33], "bf16", [0], "max", -np.inf, "bf16")
    xf = inp.bf16_bits_to_f32(x).reshape(64, 33)
    assert np.array_equal(inp.bf16_bits_to_f32(out), xf.max(axis=0))


# ---------------------------------------------------------------------------------------------
# broadcast_in_dim and add
# ---------------------------------------------------------------------------------------------
def test_broadcast_in_dim_example(orc):
    g = load_golden("broadcast_example.txt")
    out = orc.broadcast_in_dim(np.array(g["operand"], np.int32).ravel(), g["operand_dims"], "s32",
                               g["broadcast_dimensions"], g["result_dims"])
    assert out.reshape(g["result_dims"]).tolist() == g["result"]


def test_add_example_through_broadcast_operand(orc):
    g = load_golden("elementwise_examples.txt")["add"]
    lhs = np.array(g["lhs"], np.float32).ravel()
    rhs = np.array(g["rhs"], np.float32).ravel()
    chain = {"ops": ["add_bcast"], "bcast": {"data": rhs, "dims": [2, 2], "dtype": "f32",
                                             "broadcast_dimensions": [0, 1]}}
    out = orc.transpose(lhs, [2, 2], "f32", [0, 1], prologue=chain)
    assert out.reshape(2, 2).tolist() == g["result"]


def test_bcast_on_reduced_dim_with_layout(orc):
    # add(x, broadcast(b, {3})) reduced over dim 3, with the {3,2,0,1} layout: compared against numpy
    import transpose_heroes_gb300.inputs as inp

    rng = np.random.default_rng(23)
    dims = [2, 1, 3, 7]
    logical = rng.integers(-4, 4, size=dims).astype(np.float32)
    b = rng.integers(-4, 4, size=7).astype(np.float32)
    m2m = [3, 2, 0, 1]
    chain = {"ops": ["add_bcast"], "bcast": {"data": b, "dims": [7], "dtype": "f32", "broadcast_dimensions": [3]}}
    out = orc.reduce(to_physical(logical, m2m), dims, "f32", [3], "add", 0.0, "f32", m2m=m2m, prologue=chain)
    want = (logical + b.reshape(1, 1, 1, 7)).sum(axis=3)
    assert np.array_equal(out, want.ravel())
    del inp


# ---------------------------------------------------------------------------------------------
# exp / log: the spec's printed values, and correct rounding checked exactly with Decimal
# ---------------------------------------------------------------------------------------------
def test_exp_log_printed_values(orc):
    g = load_golden("elementwise_examples.txt")
    for x, y in zip(g["exp"]["x"], g["exp"]["y"]):
        assert orc.exp(x, "f64") == y
        assert orc.exp(x, "f32") == float(np.float32(y))
    for x, y in zip(g["log"]["x"], g["log"]["y"]):
        assert orc.log(x, "f64") == y
        assert orc.log(x, "f32") == float(np.float32(y))


def test_log_f32_correctly_rounded_vs_decimal(orc):
    rng = np.random.default_rng(29)
    xs = np.concatenate([rng.uniform(0.5, 2.0, 400), np.exp(rng.uniform(-80, 80, 200)),
                         1.0 + rng.uniform(-1e-3, 1e-3, 100)]).astype(np.float32)
    for x in xs:
        y = orc.log(float(x), "f32")
        lo, hi = f32_neighbors(y)
        assert exact_between_midpoints(Decimal(float(x)).ln(), y, lo, hi), x
    assert orc.log(1.0, "f32") == 0.0
    assert orc.log(0.0, "f32") == -math.inf
    assert math.isnan(orc.log(-1.0, "f32"))
    assert orc.log(math.inf, "f32") == math.inf


def test_exp_f32_and_bf16_correctly_rounded_vs_decimal(orc):
    import transpose_heroes_gb300.inputs as inp

    rng = np.random.default_rng(31)
    xs = rng.uniform(-20, 20, 300).astype(np.float32)
    for x in xs:
        y = orc.exp(float(x), "f32")
        lo, hi = f32_neighbors(y)
        assert exact_between_midpoints(Decimal(float(x)).exp(), y, lo, hi), x
    # every bf16 input in [-8, 8]: exp rounded straight to bf16
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = inp.bf16_bits_to_f32(bits)
    sel = np.isfinite(vals) & (np.abs(vals) <= 8)
    for x in vals[sel][::7]:
        y = orc.exp(float(x), "bf16")
        q = 2.0 ** (math.frexp(y)[1] - 8)  # bf16 quantum at y
        assert exact_between_midpoints(Decimal(float(x)).exp(), y, y - q if y != 2.0 ** (math.frexp(y)[1] - 1) else y - q / 2, y + q), x


def test_round_to_bf16_is_nearest_even(orc):
    rng = np.random.default_rng(37)
    for v in np.concatenate([rng.standard_normal(500) * 10, [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)]]):
        r = orc.round_to(float(v), "bf16")
        e = math.frexp(v)[1]
        q = Fraction(2) ** (e - 8)
        fv = Fraction(float(v))
        lo = (fv / q).__floor__() * q
        cands = [lo, lo + q]
        dist = [abs(fv - c) for c in cands]
        if dist[0] == dist[1]:  # tie: even significand
            want = cands[0] if (lo / q) % 2 == 0 else cands[1]
        else:
            want = cands[int(dist[1] < dist[0])]
        assert Fraction(r) == want, v


def test_bf16_spec_chain_terms(orc):
    """exp then add of a broadcast, each rounded to bf16 (the spec's types), summed exactly."""
    import transpose_heroes_gb300.inputs as inp

    rng = inp.rng(41)
    n = 257
    x = inp.normal_bf16(rng, n)
    b = inp.uniform_bf16(rng, n, -1, 1)
    chain = {"ops": ["exp", "add_bcast"], "round_each": True,
             "bcast": {"data": b, "dims": [n], "dtype": "bf16", "broadcast_dimensions": [1]}}
    out, asum = orc.reduce(x, [1, n], "bf16", [1], "add", 0.0, "f64", prologue=chain, want_abs_sum=True)
    xf, bf = inp.bf16_bits_to_f32(x), inp.bf16_bits_to_f32(b)

    def rn_bf16(fr: Fraction) -> Fraction:
        if fr == 0:
            return fr
        e = math.frexp(float(fr))[1]
        q = Fraction(2) ** (e - 8)
        lo = (fr / q).__floor__() * q
        d0, d1 = fr - lo, lo + q - fr
        if d0 == d1:
            return lo if (lo / q) % 2 == 0 else lo + q
        return lo if d0 < d1 else lo + q

    total = Fraction(0)
    for xi, bi in zip(xf, bf):
        e = Fraction(Decimal(float(xi)).exp())
        t = rn_bf16(rn_bf16(e) + Fraction(float(bi)))
        total += t
    assert out[0] == float(total)  # f64 output of an exact-enough long-double sum of bf16 terms


# ---------------------------------------------------------------------------------------------
# rounding and clamping as used by quantize
# ---------------------------------------------------------------------------------------------
def test_round_nearest_even_example(orc):
    g = load_golden("rounding_clamp_examples.txt")
    q = {"scales": [1.0], "zero_points": [0], "storage_min": -128, "storage_max": 127}
    got = [orc.quantize(q, x) for x in g["round_nearest_even"]["x"]]
    assert got == g["round_nearest_even"]["y"]
    assert got != g["round_nearest_afz"]["y"]


def test_clamp_example(orc):
    g = load_golden("rounding_clamp_examples.txt")["clamp"]
    got = []
    for lo, x, hi in zip(g["min"], g["operand"], g["max"]):
        q = {"scales": [1.0], "zero_points": [lo], "storage_min": lo, "storage_max": hi}
        got.append(orc.quantize(q, float(x - lo)))  # zero point lo: code = clamp(x - lo + lo)
    assert got == g["result"]


# ---------------------------------------------------------------------------------------------
# quantization (StableHLO Quantization; spec "Types")
# ---------------------------------------------------------------------------------------------
def test_per_tensor_example(orc):
    g = load_golden("quant_examples.txt")["per_tensor"]
    q = {"scales": [g["scale"]], "zero_points": [g["zero_point"]]}
    assert orc.dequantize(q, g["zero_code"]) == 0.0
    assert orc.quantize(q, 0.0) == g["zero_code"]
    assert orc.dequantize(q, g["zero_code"] - 100) == -1.0
    assert orc.quantize(q, -1.0) == g["zero_code"] - 100
    assert orc.quantize(q, 0.5) == g["zero_code"] + 50
    assert orc.quantize(q, 100.0) == 127 and orc.quantize(q, -100.0) == -128  # saturation


def test_per_axis_example_slices(orc):
    g = load_golden("quant_examples.txt")["per_axis"]
    dims, ax = g["dims"], g["quantization_dimension"]
    zps = np.array(g["zero_points"], np.int32)
    codes = np.zeros(dims, np.int8)
    for i in range(dims[ax]):
        codes[:, i, :] = zps[i] + 5
    spec = {"scales": np.array(g["scales"], np.float32), "zero_points": zps, "quantization_dimension": ax}
    real = orc.quant_fusion(codes.ravel(), dims, "s8", spec, [2, 1, 0], "f32").reshape(dims)
    # 5 * f32(0.2) = 1.0, 5 * f32(0.1) = 0.5, 5 * f32(0.3) = 1.5 (an exact tie, rounded to even)
    for i, want in enumerate([1.0, 0.5, 1.5]):
        assert np.all(real[:, i, :] == want)
    # each slice uses its own zero point: codes equal to the zero point give 0
    for i in range(dims[ax]):
        codes[:, i, :] = zps[i]
    real = orc.quant_fusion(codes.ravel(), dims, "s8", spec, [2, 1, 0], "f32")
    assert np.all(real == 0.0)


def test_dequant_quant_identity_all_codes(orc):
    rng = np.random.default_rng(43)
    for _ in range(20):
        s = float(np.float32(rng.uniform(0.001, 0.5)))
        z = int(rng.integers(-20, 21))
        q = {"scales": [s], "zero_points": [z]}
        for code in range(-128, 128):
            assert orc.quantize(q, orc.dequantize(q, code)) == code


def test_quant_fusion_relayout_vs_numpy(orc):
    import transpose_heroes_gb300.inputs as inp

    f = inp.small("quant_relayout", n0=37, n1=29)
    out = orc.quant_fusion(f.data, f.dims, "s8", f.in_q, f.out_m2m, "s8", out_q=f.out_q)
    q = f.data.reshape(f.dims).astype(np.int32)
    sc, zp = f.in_q["scales"], f.in_q["zero_points"]
    real = (sc[None, :] * (q - zp[None, :]).astype(np.float32)).astype(np.float32)  # f32 multiply
    ratio = (real / np.float32(0.05)).astype(np.float32)                               # f32 divide
    want = np.clip(np.rint(ratio), -128, 127).astype(np.int8)                          # ties to even
    assert np.array_equal(from_physical(out, f.dims, f.out_m2m), want)


# ---------------------------------------------------------------------------------------------
# tanh, constants and the loop fusion (XLA:GPU Emitters, "Loop emitter": the GELU function)
# ---------------------------------------------------------------------------------------------
FORMATS = {"bf16": (8, -126, 127), "f16": (11, -14, 15), "f32": (24, -126, 127)}


def round_fraction(q: Fraction, fmt: str) -> float:
    """Nearest value of the binary format to the exact rational q, ties to even, gradual underflow,
    overflow to infinity (test-side, written independently of the oracle)."""
    prec, emin, emax = FORMATS[fmt]
    if q == 0:
        return 0.0
    sign, a = (-1, -q) if q < 0 else (1, q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    lead = max(e, emin)
    quantum = Fraction(2) ** (lead - prec + 1)
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * quantum
    if r > Fraction(2) ** emax * (2 - Fraction(2) ** (1 - prec)):
        return sign * math.inf
    return sign * float(r)


def decimal_tanh(x: float) -> Fraction:
    """tanh(x) to ~60 significant digits as an exact rational (series near 0, exp form elsewhere)."""
    d = Decimal(x)
    if abs(d) < Decimal("1e-6"):
        t = d - d ** 3 / 3 + 2 * d ** 5 / 15 - 17 * d ** 7 / 315
    else:
        em = (-2 * abs(d)).exp()  # e^{-2|x|}: no overflow for large |x|
        t = (1 - em) / (1 + em)
        t = t if d > 0 else -t
    return Fraction(t)


def bf16_values():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    return bits.view(np.float32)


def f16_values():
    return np.arange(1 << 16, dtype=np.uint16).view(np.float16).astype(np.float32)


def chain_1d(orc, data, dtype, ops):
    n = len(data)
    return orc.transpose(data, [n], dtype, [0], prologue={"ops": ops, "round_each": True})


def test_gelu_constants_match_the_printed_mlir(orc):
    g = load_golden("gelu_loop_fusion.txt")
    for c, printed in zip(g["hlo_constants"], g["printed_bf16"]):
        # the MLIR prints a bf16 constant with a short decimal that reads back as the same bf16 value
        v = orc.round_to(c, "bf16")
        assert v == orc.round_to(float(printed), "bf16") == round_fraction(Fraction(printed), "bf16")
        assert v == round_fraction(Fraction(c), "bf16")


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_tanh_every_16bit_input_correctly_rounded(orc, fmt):
    vals = bf16_values() if fmt == "bf16" else f16_values()
    if fmt == "bf16":
        got = chain_1d(orc, (vals.view(np.uint32) >> 16).astype(np.uint16), "bf16", ["tanh"])
        got = (got.astype(np.uint32) << 16).view(np.float32)
    else:  # f16 travels as its bit pattern
        got = chain_1d(orc, np.arange(1 << 16, dtype=np.uint16), "f16", ["tanh"])
        got = np.asarray(got, dtype=np.uint16).view(np.float16).astype(np.float32)
    bad = 0
    for x, y in zip(vals, got):
        x = float(x)
        if math.isnan(x):
            bad += not math.isnan(float(y))
            continue
        if math.isinf(x):
            bad += float(y) != math.copysign(1.0, x)
            continue
        want = x if x == 0 else round_fraction(decimal_tanh(x), fmt)  # tanh(+-0) = +-0
        bad += (float(y) != want) or (math.copysign(1.0, float(y)) != math.copysign(1.0, want))
    assert bad == 0


def test_tanh_f32_sample_correctly_rounded(orc):
    g = np.random.default_rng(5)
    x = np.concatenate([g.uniform(-6, 6, 1500), g.uniform(-1e-3, 1e-3, 300), [0.5, -2.0, 1e-20, 9.0]])
    x = x.astype(np.float32)
    got = chain_1d(orc, x, "f32", ["tanh"])
    for xi, yi in zip(x, got):
        assert float(yi) == round_fraction(decimal_tanh(float(xi)), "f32"), float(xi)


@pytest.mark.parametrize("fmt", ["bf16", "f32"])
def test_constant_and_input_ops_exact(orc, fmt):
    """v <- x*x + c, * d, + x, * x: each step the exact rational result rounded to the format."""
    g = np.random.default_rng(6)
    x = g.standard_normal(500).astype(np.float32) * np.float32(3)
    c, d = 0.1, -1.7
    if fmt == "bf16":
        xb = (x.view(np.uint32) >> 16).astype(np.uint16)  # truncation makes valid bf16 values
        xs = (xb.astype(np.uint32) << 16).view(np.float32)
        got = chain_1d(orc, xb, "bf16", ["mul_input", ["add_const", c], ["mul_const", d], "add_input", "mul_input"])
        got = (got.astype(np.uint32) << 16).view(np.float32)
    else:
        xs = x
        got = chain_1d(orc, x, "f32", ["mul_input", ["add_const", c], ["mul_const", d], "add_input", "mul_input"])
    cq, dq = Fraction(round_fraction(Fraction(c), fmt)), Fraction(round_fraction(Fraction(d), fmt))
    for xi, yi in zip(xs, got):
        xq = Fraction(float(xi))
        v = Fraction(round_fraction(xq * xq, fmt))
        v = Fraction(round_fraction(v + cq, fmt))
        v = Fraction(round_fraction(v * dq, fmt))
        v = Fraction(round_fraction(v + xq, fmt))
        want = round_fraction(v * xq, fmt)
        assert float(yi) == want


def gelu_reference(x: float) -> float:
    """The HLO's ops on exact rationals, each rounded to bf16 (test-side)."""
    def r(q):
        return Fraction(round_fraction(q, "bf16"))
    c3, c2, c1, c0 = (r(Fraction(v)) for v in (0.044708, 0.79785, 1.0, 0.5))
    xq = Fraction(x)
    sq = r(xq * xq)
    cube = r(sq * xq)
    m3 = r(cube * c3)
    a1 = r(xq + m3)
    m2 = r(a1 * c2)
    th = r(decimal_tanh(float(m2)))
    a0 = r(th + c1)
    m1 = r(a0 * c0)
    out = round_fraction(xq * m1, "bf16")
    # m1 >= 0 (tanh >= -1), so an IEEE zero product carries the sign of x
    return math.copysign(0.0, x) if out == 0 else out


def test_gelu_chain_against_exact_evaluation(orc):
    g = load_golden("gelu_loop_fusion.txt")
    ops = [tuple(o) if isinstance(o, list) else o for o in g["ops"]]
    vals = bf16_values()
    finite = vals[np.isfinite(vals) & (np.abs(vals) < 1e4)]
    sample = np.concatenate([finite[::13], np.float32([0.0, -0.0, 1.0, -1.0, 8.0, -8.0, 0.5])])
    xb = (sample.view(np.uint32) >> 16).astype(np.uint16)
    got = (chain_1d(orc, xb, "bf16", ops).astype(np.uint32) << 16).view(np.float32)
    for xi, yi in zip(sample, got):
        want = gelu_reference(float(xi))
        assert float(yi) == want and math.copysign(1.0, float(yi)) == math.copysign(1.0, want), float(xi)
    # closed forms: gelu(x) = x once tanh rounds to 1; gelu(-x) = -0 once it rounds to -1
    big = (np.float32([4.0, 8.0, 100.0]).view(np.uint32) >> 16).astype(np.uint16)
    out = (chain_1d(orc, big, "bf16", ops).astype(np.uint32) << 16).view(np.float32)
    assert list(out) == [4.0, 8.0, 100.0]
    neg = (np.float32([-8.0, -100.0]).view(np.uint32) >> 16).astype(np.uint16)
    out = (chain_1d(orc, neg, "bf16", ops).astype(np.uint32) << 16).view(np.float32)
    assert all(v == 0 and math.copysign(1.0, float(v)) < 0 for v in out)


# ---------------------------------------------------------------------------------------------
# variadic reduce with the max/argmax body (XLA Operation Semantics, "Variadic Reduce")
# ---------------------------------------------------------------------------------------------
def test_argmax_closed_forms(orc):
    ninf = -math.inf
    # equal maxima keep the last index (value >= max replaces)
    v, i = orc.reduce_max_argmax(np.float32([1, 3, 2, 3, 0]), [5], "f32", [0], ninf, -1)
    assert (v[0], i[0]) == (3.0, 3)
    # NaN never compares >= max, so it is never selected
    v, i = orc.reduce_max_argmax(np.float32([np.nan, 2, np.nan, 1]), [4], "f32", [0], ninf, -1)
    assert (v[0], i[0]) == (2.0, 1)
    # an init above every value survives with its index; an init equal to the max is replaced
    v, i = orc.reduce_max_argmax(np.float32([1, 2, 3]), [3], "f32", [0], 7.0, 42)
    assert (v[0], i[0]) == (7.0, 42)
    v, i = orc.reduce_max_argmax(np.float32([1, 3, 2]), [3], "f32", [0], 3.0, 42)
    assert (v[0], i[0]) == (3.0, 1)
    # an empty reduced dimension yields the init values
    v, i = orc.reduce_max_argmax(np.zeros(0, np.float32), [4, 0], "f32", [1], ninf, -5)
    assert list(v) == [ninf] * 4 and list(i) == [-5] * 4
    # a ramp: the last position
    v, i = orc.reduce_max_argmax(np.arange(10, dtype=np.float32), [10], "f32", [0], ninf, -1)
    assert (v[0], i[0]) == (9.0, 9)


@pytest.mark.parametrize("dimsred", [[1], [0], [0, 2], [2, 1]])
def test_argmax_against_numpy_last_maximum(orc, dimsred):
    """Random small integers (many ties), explicit K = a random permutation: the answer is K at the
    last position, in the lexicographic walk of the reduced dims, that holds the maximum."""
    g = np.random.default_rng(21)
    dims = [5, 7, 6]
    v = g.integers(-3, 4, size=dims).astype(np.float32)
    k = g.permutation(int(np.prod(dims))).astype(np.int32).reshape(dims)
    for m2m in ([2, 1, 0], [0, 2, 1]):
        vals, idx = orc.reduce_max_argmax(to_physical(v, m2m), dims, "f32", dimsred, -math.inf, -1, m2m=m2m,
                                          indices=to_physical(k, m2m), idx_m2m=m2m)
        kept = [d for d in range(3) if d not in dimsred]
        order = kept + sorted(dimsred)  # reduced dims in increasing order: the lexicographic walk
        vv = np.transpose(v, order).reshape([dims[d] for d in kept] + [-1])
        kk = np.transpose(k, order).reshape([dims[d] for d in kept] + [-1])
        n = vv.shape[-1]
        last = n - 1 - np.argmax(vv[..., ::-1], axis=-1)
        want_v = np.take_along_axis(vv, last[..., None], -1)[..., 0]
        want_k = np.take_along_axis(kk, last[..., None], -1)[..., 0]
        # outputs in the default layout: row-major over the kept dims in their logical order
        assert np.array_equal(vals, want_v.ravel())
        assert np.array_equal(idx, want_k.ravel())


# ---------------------------------------------------------------------------------------------
# quantized elementwise binary ops (StableHLO Specification, add/divide/maximum/minimum/multiply on
# quantized types: dequantize_op_quantize)
# ---------------------------------------------------------------------------------------------
def _pt(scale, zp):
    return {"scales": np.float32([scale]), "zero_points": np.int32([zp]), "quantization_dimension": None}


ALL_CODES = np.arange(-128, 128, dtype=np.int8)


def test_quant_binary_invariants(orc):
    q = _pt(0.3, 0)  # the pages' quantized-add test type !quant.uniform<i8:f32, 0.3>
    a = np.repeat(ALL_CODES, 256)
    b = np.tile(ALL_CODES, 256)
    dims = [a.size]
    zero = np.zeros_like(a)
    # x + 0 and max(x, x) requantized with the same parameters give x back
    assert np.array_equal(orc.quant_binary("add", a, zero, dims, q, q, q), a)
    assert np.array_equal(orc.quant_binary("maximum", a, a, dims, q, q, q), a)
    assert np.array_equal(orc.quant_binary("minimum", a, a, dims, q, q, q), a)
    # commutative ops
    for op in ("add", "multiply", "maximum", "minimum"):
        assert np.array_equal(orc.quant_binary(op, a, b, dims, q, _pt(0.7, 3), _pt(0.2, -5)),
                              orc.quant_binary(op, b, a, dims, _pt(0.7, 3), q, _pt(0.2, -5)))
    # max/min of equal parameters pick one operand's code
    mx = orc.quant_binary("maximum", a, b, dims, q, q, q)
    assert np.array_equal(mx, np.maximum(a, b))
    assert np.array_equal(orc.quant_binary("minimum", a, b, dims, q, q, q), np.minimum(a, b))
    # x / x = 1 exactly (for x != zero point); 1 / 0.25 = 4
    nz = a[a != 0]
    assert np.all(orc.quant_binary("divide", nz, nz, [nz.size], q, q, _pt(0.25, 0)) == 4)
    # saturation: 127 * 0.3 * 127 * 0.3 / 0.01 is far above the storage range
    assert orc.quant_binary("multiply", np.int8([127]), np.int8([127]), [1], q, q, _pt(0.01, 0))[0] == 127
    # 0 / 0 is NaN, which quantizes to the zero point
    assert orc.quant_binary("divide", np.int8([0]), np.int8([0]), [1], q, q, _pt(0.5, 7))[0] == 7


@pytest.mark.parametrize("op", ["add", "divide", "maximum", "minimum", "multiply"])
def test_quant_binary_exact_steps(orc, op):
    """Each step on exact rationals with the rounding the definition prescribes: the f32 product
    scale * (q - zp), the f32 op, the f32 quotient by the result scale, ties to even, clamp."""
    g = np.random.default_rng(7 + len(op))
    a = g.integers(-128, 128, 400).astype(np.int8)
    b = g.integers(-128, 128, 400).astype(np.int8)
    sl, zl, sr, zr, so, zo = 0.0371, 4, 0.113, -9, 0.09, 2
    got = orc.quant_binary(op, a, b, [400], _pt(sl, zl), _pt(sr, zr), _pt(so, zo))
    f = lambda v: Fraction(round_fraction(Fraction(float(np.float32(v))), "f32"))
    S = {k: f(v) for k, v in dict(sl=sl, sr=sr, so=so).items()}
    for x, y, r in zip(a, b, got):
        dl = Fraction(round_fraction(S["sl"] * (int(x) - zl), "f32"))
        dr = Fraction(round_fraction(S["sr"] * (int(y) - zr), "f32"))
        if op == "add":
            v = dl + dr
        elif op == "multiply":
            v = dl * dr
        elif op == "maximum":
            v = max(dl, dr)
        elif op == "minimum":
            v = min(dl, dr)
        else:
            if dr == 0:
                want = zo if dl == 0 else (127 if dl > 0 else -128)
                assert r == want
                continue
            v = dl / dr
        v = Fraction(round_fraction(v, "f32"))
        ratio = Fraction(round_fraction(v / S["so"], "f32"))
        fl = ratio.numerator // ratio.denominator
        rem = ratio - fl
        if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
            fl += 1
        assert r == max(-128, min(127, fl + zo))


# ---------------------------------------------------------------------------------------------
# f32 intermediates for 16-bit chains (round_intermediates = 0). This is the emitter's lowering of a
# bf16/f16 op through f32 (XLA:GPU Emitters, "Loop emitter": fpext -> f32 op -> fptrunc) with the
# fptrunc/fpext pair between two fused ops left out: every op is the correctly rounded f32 operation,
# the value is rounded to the element type once, where the chain's result is stored. A constant keeps
# the type of its HLO constant instruction, the element type (StableHLO Specification, "constant"):
# constant(0.1) of bf16 is the bf16 value 0.10009765625 whichever precision the ops run in.
# ---------------------------------------------------------------------------------------------
def _exact_unary(name: str, v: Fraction) -> Fraction:
    """The exact value (to ~80 digits) of op(v) for an f32 value v, as a rational."""
    if name == "exp":
        return Fraction(Decimal(float(v)).exp())
    if name == "log":
        return Fraction(Decimal(float(v)).ln())
    if name == "tanh":
        return decimal_tanh(float(v))
    raise ValueError(name)


def _chain_f32_mode(ops, x: float, fmt: str, const_fmt: str) -> float:
    """Test-side evaluation of a chain with f32 intermediates: each op's exact result rounded to f32,
    constants rounded to const_fmt, one final rounding to fmt."""
    xq = Fraction(x)
    v = xq
    for op in ops:
        if isinstance(op, (tuple, list)):
            name, c = op
            cq = Fraction(round_fraction(Fraction(c), const_fmt))
            v = v + cq if name == "add_const" else v * cq
        elif op in ("exp", "log", "tanh"):
            v = _exact_unary(op, v)
        elif op == "abs":
            v = abs(v)
        elif op == "neg":
            v = -v
        elif op == "add_input":
            v = v + xq
        elif op == "mul_input":
            v = v * xq
        v = Fraction(round_fraction(v, "f32"))
    return round_fraction(v, fmt)


def _bits_of(vals, fmt):
    if fmt == "bf16":
        return (vals.view(np.uint32) >> 16).astype(np.uint16)
    return vals.astype(np.float16).view(np.uint16)


def _vals_of(bits, fmt):
    if fmt == "bf16":
        return (np.asarray(bits, np.uint32) << 16).view(np.float32)
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float32)


F32_MODE_CHAINS = [
    ["exp", ("add_const", 0.1), ("mul_const", -1.7), "tanh"],
    ["abs", ("add_const", 0.01), "log", "mul_input", "neg"],
]


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
@pytest.mark.parametrize("ops", F32_MODE_CHAINS, ids=["exp-const-tanh", "abs-log-input"])
def test_chain_with_f32_intermediates_exact(orc, fmt, ops):
    g = np.random.default_rng(29)
    x = g.uniform(-6, 6, 400).astype(np.float32)
    bits = _bits_of(x, fmt)  # bf16 by truncation, f16 by numpy's nearest: both valid 16-bit values
    xs = _vals_of(bits, fmt)
    got = orc.transpose(bits, [len(bits)], fmt, [0], prologue={"ops": ops, "round_each": False})
    got = _vals_of(got, fmt)
    differs_from_spec_types = differs_from_f32_consts = 0
    spec = _vals_of(orc.transpose(bits, [len(bits)], fmt, [0], prologue={"ops": ops, "round_each": True}), fmt)
    for xi, yi, si in zip(xs, got, spec):
        want = _chain_f32_mode(ops, float(xi), fmt, const_fmt=fmt)
        assert float(yi) == want, (float(xi), float(yi), want)
        differs_from_spec_types += float(si) != want
        differs_from_f32_consts += _chain_f32_mode(ops, float(xi), fmt, const_fmt="f32") != want
    # the pin discriminates: per-op rounding to the element type, and f32 constants, each change results
    assert differs_from_spec_types > 0
    assert differs_from_f32_consts > 0


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_reduce_terms_with_f32_intermediates_exact(orc, fmt):
    """exp then add of a broadcast operand with f32 intermediates: each term is f32(f32(exp x) + b),
    never rounded to the 16-bit type, and the terms are summed (the f64 oracle sum is exact here)."""
    import transpose_heroes_gb300.inputs as inp

    rng = inp.rng(43)
    n = 300
    if fmt == "bf16":
        x = inp.normal_bf16(rng, n)
        b = inp.uniform_bf16(rng, n, -1, 1)
    else:
        x = rng.standard_normal(n).astype(np.float16).view(np.uint16)
        b = rng.uniform(-1, 1, n).astype(np.float16).view(np.uint16)
    chain = {"ops": ["exp", "add_bcast"], "round_each": False,
             "bcast": {"data": b, "dims": [n], "dtype": fmt, "broadcast_dimensions": [1]}}
    out = orc.reduce(x, [1, n], fmt, [1], "add", 0.0, "f64", prologue=chain)
    total = total_spec = Fraction(0)
    for xi, bi in zip(_vals_of(x, fmt), _vals_of(b, fmt)):
        e = Fraction(round_fraction(Fraction(Decimal(float(xi)).exp()), "f32"))
        total += Fraction(round_fraction(e + Fraction(float(bi)), "f32"))
        e16 = Fraction(round_fraction(Fraction(Decimal(float(xi)).exp()), fmt))
        total_spec += Fraction(round_fraction(e16 + Fraction(float(bi)), fmt))
    assert out[0] == float(total)
    assert float(total) != float(total_spec)  # the two readings give different sums


def test_reduce_init_is_a_value_of_the_input_type(orc):
    """reduce (C2): init_values has the inputs' element type, so init 0.1 on bf16 inputs is the bf16
    value 0.10009765625 (on f16 0.0999755859375, on f32 the f32 nearest 0.1)."""
    for fmt, want in [("bf16", 0.10009765625), ("f16", 0.0999755859375), ("f32", float(np.float32(0.1)))]:
        zeros = np.zeros(4, dtype=np.float32 if fmt == "f32" else np.uint16)
        out = orc.reduce(zeros, [1, 4], fmt, [1], "add", 0.1, "f64")
        assert out[0] == want == round_fraction(Fraction(0.1), fmt)
        empty = orc.reduce(np.zeros(0, np.float32 if fmt == "f32" else np.uint16), [3, 0], fmt, [1], "max", 0.1,
                           "f64")
        assert list(empty) == [want] * 3


# ---------------------------------------------------------------------------------------------
# quantize: round, then add the zero point, then clamp (the reading of the missing uniform_quantize
# section; the other order, adding the zero point before rounding, changes exact ties when the zero
# point is odd). And the float ops between dequantize and quantize, pinned step by step.
# ---------------------------------------------------------------------------------------------
def test_quantize_adds_the_zero_point_after_rounding(orc):
    odd = {"scales": [1.0], "zero_points": [1]}
    assert orc.quantize(odd, 2.5) == 3    # RNE(2.5) = 2, + 1; zero point first: RNE(3.5) = 4
    assert orc.quantize(odd, 3.5) == 5    # RNE(3.5) = 4, + 1; zero point first: RNE(4.5) = 4
    assert orc.quantize(odd, -0.5) == 1   # RNE(-0.5) = -0, + 1; zero point first: RNE(0.5) = 0
    neg = {"scales": [1.0], "zero_points": [-3]}
    assert orc.quantize(neg, 0.5) == -3   # RNE(0.5) = 0, - 3; zero point first: RNE(-2.5) = -2
    # the clamp comes last: 126.5 -> 126 + 1 = 127; 127.5 -> 128 + 1 -> clamped to 127
    assert orc.quantize(odd, 126.5) == 127 and orc.quantize(odd, 127.5) == 127
    assert orc.quantize({"scales": [0.5], "zero_points": [1]}, 1.25) == 3  # 1.25/0.5 = 2.5 -> 2, + 1


def _rne_int(q: Fraction) -> int:
    fl = q.numerator // q.denominator
    rem = q - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


@pytest.mark.parametrize("out_kind", ["s8", "f32"])
def test_quant_fusion_float_ops_chain_exact(orc, out_kind):
    """dequantize (per-axis on dim 1) -> abs, neg, exp, *1.5, +(-0.25) in f32 -> relayout {1,0} -> {0,1}
    -> quantize (0.01, zero point 3) or the f32 value, each step on exact rationals rounded to f32."""
    g = np.random.default_rng(23)
    n0, n1 = 12, 20
    q = g.integers(-128, 128, size=(n0, n1)).astype(np.int8)
    scales = g.uniform(0.001, 0.01, n1).astype(np.float32)
    zps = g.integers(-20, 21, n1).astype(np.int32)
    in_q = {"scales": scales, "zero_points": zps, "quantization_dimension": 1}
    out_q = {"scales": [0.01], "zero_points": [3]} if out_kind == "s8" else None
    ops = ["abs", "neg", "exp", ("mul_const", 1.5), ("add_const", -0.25)]
    out = orc.quant_fusion(q.ravel(), [n0, n1], "s8", in_q, [0, 1], out_kind, out_q=out_q,
                           float_ops={"ops": ops})
    s_out = Fraction(float(np.float32(0.01)))

    def f32(v):
        return Fraction(round_fraction(v, "f32"))

    for i in range(n0):
        for j in range(n1):
            v = f32(Fraction(float(scales[j])) * (int(q[i, j]) - int(zps[j])))
            v = -abs(v)
            v = f32(Fraction(Decimal(float(v)).exp()))
            v = f32(v * f32(Fraction(1.5)))
            v = f32(v + f32(Fraction(-0.25)))
            got = out[j * n0 + i]  # layout {0,1}: dimension 0 is minor
            if out_kind == "f32":
                assert Fraction(float(got)) == v
            else:
                code = min(127, max(-128, _rne_int(f32(v / s_out)) + 3))
                assert int(got) == code, (i, j)


# ---------------------------------------------------------------------------------------------
# quantized broadcast_in_dim and reshape (StableHLO Specification, "broadcast_in_dim" C1, C6;
# "reshape" C1-C3): stored codes move like plain elements, the parameters follow the constraints
# ---------------------------------------------------------------------------------------------
def _dequant_logical(codes, dims, params):
    """Test-side dequantize of a logical (row-major) code array with numpy f32 arithmetic."""
    c = np.asarray(codes, np.int32).reshape(dims)
    s = np.asarray(params["scales"], np.float32)
    z = np.asarray(params["zero_points"], np.int32)
    qd = params.get("quantization_dimension")
    if qd is None:
        return (s[0] * (c - z[0]).astype(np.float32)).astype(np.float32)
    shape = [1] * len(dims)
    shape[qd] = dims[qd]
    return (s.reshape(shape) * (c - z.reshape(shape)).astype(np.float32)).astype(np.float32)


def test_quant_broadcast_in_dim_example_per_axis(orc):
    """The spec's example [[1, 2, 3]] -> tensor<2x3x2> with broadcast_dimensions [2, 1], quantized per
    axis along operand dimension 1 with the quantization page's {0.2:20, 0.1:10, 0.3:30}: the codes are
    the printed result and the result is per-axis along broadcast_dimensions[1] = 1 (C6) with the same
    parameters."""
    g = load_golden("broadcast_example.txt")
    qa = load_golden("quant_examples.txt")["per_axis"]
    q = {"scales": np.float32(qa["scales"]), "zero_points": np.int32(qa["zero_points"]), "quantization_dimension": 1}
    codes, params = orc.quant_broadcast_in_dim(np.int8(g["operand"]).ravel(), g["operand_dims"], q,
                                               g["broadcast_dimensions"], g["result_dims"])
    assert codes.reshape(g["result_dims"]).tolist() == g["result"]
    assert params["quantization_dimension"] == 1
    assert params["scales"].tolist() == np.float32(qa["scales"]).tolist()
    assert params["zero_points"].tolist() == qa["zero_points"]
    # the real values are broadcast: result[i, j, k] = real(operand[0, j])
    real_in = _dequant_logical(np.int8(g["operand"]).ravel(), g["operand_dims"], q)
    real_out = _dequant_logical(codes, g["result_dims"], params)
    for i in range(2):
        for j in range(3):
            for k in range(2):
                assert real_out[i, j, k] == real_in[0, j]


def test_quant_broadcast_in_dim_unit_quantized_dimension(orc):
    """C6: when dim(operand, qd) = 1, the single (scale, zero_point) is repeated along the result's
    quantization dimension; a per-tensor operand stays per-tensor (C1)."""
    q = {"scales": np.float32([0.5]), "zero_points": np.int32([2]), "quantization_dimension": 0}
    codes, params = orc.quant_broadcast_in_dim(np.int8([7, -3, 1]), [1, 3], q, [2, 1], [4, 3, 5])
    assert params["quantization_dimension"] == 2
    assert params["scales"].tolist() == [0.5] * 5 and params["zero_points"].tolist() == [2] * 5
    assert np.array_equal(codes.reshape(4, 3, 5), np.broadcast_to(np.int8([7, -3, 1])[None, :, None], (4, 3, 5)))
    pt = {"scales": np.float32([0.25]), "zero_points": np.int32([-1])}
    _, params = orc.quant_broadcast_in_dim(np.int8([7, -3, 1]), [1, 3], pt, [2, 1], [4, 3, 5])
    assert params["quantization_dimension"] is None and params["scales"].tolist() == [0.25]


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_quant_broadcast_in_dim_commutes_with_dequantize(orc, seed):
    """dequantize(broadcast_in_dim(q)) = broadcast_in_dim(dequantize(q)) exactly, on random shapes,
    broadcast dimensions, layouts and per-axis dimensions (brute force against numpy)."""
    g = np.random.default_rng(seed)
    rank_in = int(g.integers(1, 4))
    rank_out = rank_in + int(g.integers(0, 3))
    bdims = sorted(g.choice(rank_out, size=rank_in, replace=False).tolist())
    if seed == 3:
        bdims = bdims[::-1]  # broadcast_dimensions need not be increasing
    out_dims = [int(v) for v in g.integers(1, 5, size=rank_out)]
    dims = [1 if g.random() < 0.3 else out_dims[b] for b in bdims]
    qd = int(g.integers(0, rank_in))
    q = {"scales": g.uniform(0.01, 0.5, dims[qd]).astype(np.float32),
         "zero_points": g.integers(-20, 21, dims[qd]).astype(np.int32), "quantization_dimension": qd}
    codes = g.integers(-128, 128, size=dims).astype(np.int8)
    in_m2m = g.permutation(rank_in).tolist()
    out_m2m = g.permutation(rank_out).tolist()
    out, params = orc.quant_broadcast_in_dim(to_physical(codes, in_m2m), dims, q, bdims, out_dims, m2m=in_m2m,
                                             out_m2m=out_m2m)
    out_logical = from_physical(out, out_dims, out_m2m)
    assert params["quantization_dimension"] == bdims[qd]
    real_in = _dequant_logical(codes.ravel(), dims, q)
    real_out = _dequant_logical(out_logical.ravel(), out_dims, params)
    # numpy broadcast of the dequantized operand: move operand dim d to result dim bdims[d]
    expand = np.zeros([1] * rank_out, np.float32) + 0
    shape = [1] * rank_out
    order = np.argsort(bdims)
    moved = np.transpose(real_in, order).reshape([dims[d] for d in order])
    for d in range(rank_in):
        shape[bdims[d]] = dims[d]
    want = np.broadcast_to(moved.reshape(shape) + expand, out_dims)
    assert np.array_equal(real_out, want)


def test_reshape_example(orc):
    g = load_golden("reshape_example.txt")
    out = orc.reshape(np.int32(g["operand"]).ravel(), g["operand_dims"], g["result_dims"], "s32")
    assert out.reshape(g["result_dims"]).tolist() == g["result"]


def test_quant_reshape_per_axis_rules(orc):
    """C3 on the quantization page's t[4, 3, 2] (per-axis along 1): [2, 2, 3, 2] keeps the axis (before 4,
    size 3, after 2) as dimension 2; [12, 2] and [4, 6] do not; a per-tensor operand has no axis."""
    qa = load_golden("quant_examples.txt")["per_axis"]
    q = {"scales": np.float32(qa["scales"]), "zero_points": np.int32(qa["zero_points"]), "quantization_dimension": 1}
    g = np.random.default_rng(7)
    codes = g.integers(-128, 128, size=qa["dims"]).astype(np.int8)
    out = orc.reshape(codes.ravel(), qa["dims"], [2, 2, 3, 2], "s8", q=q, result_qdim=2)
    assert np.array_equal(out, codes.ravel())  # default layouts: the same bytes
    rq = dict(q, quantization_dimension=2)
    assert np.array_equal(_dequant_logical(out, [2, 2, 3, 2], rq).ravel(), _dequant_logical(codes.ravel(), qa["dims"], q).ravel())
    for bad_dims, bad_qd in [([12, 2], 0), ([4, 6], 1), ([2, 2, 3, 2], 1), ([4, 3, 2], 2)]:
        with pytest.raises(ValueError):
            orc.reshape(codes.ravel(), qa["dims"], bad_dims, "s8", q=q, result_qdim=bad_qd)
    with pytest.raises(ValueError):  # C2: the element count is kept
        orc.reshape(codes.ravel(), qa["dims"], [5, 5], "s8")
    pt = {"scales": np.float32([0.1]), "zero_points": np.int32([0])}
    assert np.array_equal(orc.reshape(codes.ravel(), qa["dims"], [24], "s8", q=pt, result_qdim=-1), codes.ravel())


@pytest.mark.parametrize("seed", [1, 2])
def test_reshape_with_layouts_vs_numpy(orc, seed):
    g = np.random.default_rng(seed)
    dims, out_dims = [3, 4, 5], [6, 10]
    x = g.integers(-1000, 1000, size=dims).astype(np.int32)
    for in_m2m in all_layouts(3):
        for out_m2m in ([1, 0], [0, 1]):
            out = orc.reshape(to_physical(x, in_m2m), dims, out_dims, "s32", m2m=in_m2m, out_m2m=out_m2m)
            assert np.array_equal(from_physical(out, out_dims, out_m2m), x.reshape(out_dims))
