"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every entry point the header
declares, and rejects invalid arguments (the spec's constraints) before touching the device."""

import ctypes
import os
import re

import numpy as np
import pytest

from conftest import ROOT

import transpose_heroes_gb300 as hf
from transpose_heroes_gb300 import build as hbuild

HEADER = os.path.join(ROOT, "include", "hlo_fusion.h")
FAKE_IN, FAKE_OUT = 0x100000, 0x900000  # never dereferenced: every call below fails validation first


@pytest.fixture(scope="module")
def lib():
    hbuild.build()
    return hf.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:hlo_status|size_t|int32_t|int64_t|const char\*)\s+(hlo_\w+)\s*\(", text, re.M)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(hf.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert "sm_103a" in hf.version()


def test_library_is_built_for_sm_103a_only():
    text = open(hbuild.__file__).read()
    assert "arch=compute_103a,code=sm_103a" in text


def _status(call):
    with pytest.raises(hf.HloError) as e:
        call()
    return e.value.status, str(e.value)


def test_reduce_validation(lib):
    x = FAKE_IN
    out = FAKE_OUT
    # C5: repeated dimension
    st, msg = _status(lambda: hf.reduce_fusion(x, [4, 5], "f32", [1, 1], "add", 0.0, out, "f32", stream=0))
    assert st == 1 and "C5" in msg
    # C4: dimension out of range
    st, msg = _status(lambda: hf.reduce_fusion(x, [4, 5], "f32", [2], "add", 0.0, out, "f32", stream=0))
    assert st == 1 and "C4" in msg
    # layout not a permutation
    st, msg = _status(lambda: hf.reduce_fusion(x, [4, 5], "f32", [1], "add", 0.0, out, "f32", in_m2m=[0, 0],
                                               stream=0))
    assert st == 1 and "minor_to_major" in msg
    # integer input is not supported by the reduce kernels
    st, _ = _status(lambda: hf.reduce_fusion(x, [4, 5], "s32", [1], "add", 0.0, out, "f32", stream=0))
    assert st == 2
    # input and output overlap
    st, msg = _status(lambda: hf.reduce_fusion(x, [4, 5], "f32", [1], "add", 0.0, x + 8, "f32", stream=0))
    assert st == 1 and "overlap" in msg


def test_reduce_output_shape_rule_c7(lib):
    a = hf.make_array([4, 5], None, "f32")
    o = hf.make_array([5], None, "f32")  # kept dim 0 has size 4, not 5
    dims = (ctypes.c_int64 * 1)(1)
    st = lib.hlo_reduce_fusion(ctypes.byref(a), FAKE_IN, None, dims, 1, 0, 0.0, 0, ctypes.byref(o), FAKE_OUT,
                               None, 0, 0)
    assert st == 1 and "C7" in hf.last_error()
    # f64 accumulation is not implemented
    o = hf.make_array([4], None, "f32")
    st = lib.hlo_reduce_fusion(ctypes.byref(a), FAKE_IN, None, dims, 1, 0, 0.0, 3, ctypes.byref(o), FAKE_OUT,
                               None, 0, 0)
    assert st == 2


def test_broadcast_validation(lib):
    bad_c5 = {"ops": ["add_bcast"], "bcast": {"tensor": 0x5000, "dims": [7], "dtype": "f32",
                                               "broadcast_dimensions": [1]}}
    st, msg = _status(lambda: hf.reduce_fusion(FAKE_IN, [4, 5], "f32", [1], "add", 0.0, FAKE_OUT, "f32",
                                               prologue=bad_c5, stream=0))
    assert st == 1 and "C5" in msg
    bad_c3 = {"ops": ["add_bcast"], "bcast": {"tensor": 0x5000, "dims": [5], "dtype": "f32",
                                               "broadcast_dimensions": [2]}}
    st, msg = _status(lambda: hf.reduce_fusion(FAKE_IN, [4, 5], "f32", [1], "add", 0.0, FAKE_OUT, "f32",
                                               prologue=bad_c3, stream=0))
    assert st == 1 and "C3" in msg
    bad_type = {"ops": ["add_bcast"], "bcast": {"tensor": 0x5000, "dims": [5], "dtype": "bf16",
                                                 "broadcast_dimensions": [1]}}
    st, msg = _status(lambda: hf.reduce_fusion(FAKE_IN, [4, 5], "f32", [1], "add", 0.0, FAKE_OUT, "f32",
                                               prologue=bad_type, stream=0))
    assert st == 1 and "C1" in msg


def test_transpose_validation(lib):
    st, msg = _status(lambda: hf.transpose_fusion(FAKE_IN, [3, 4], "f32", [0, 0], FAKE_OUT, stream=0))
    assert st == 1 and "permutation" in msg
    st, msg = _status(lambda: hf.transpose_fusion(FAKE_IN, [3, 4], "f32", [1, 0], FAKE_OUT, self_add=True, stream=0))
    assert st == 1 and "self-add" in msg
    st, _ = _status(lambda: hf.transpose_fusion(FAKE_IN, [3, 4], "s8", [1, 0], FAKE_OUT,
                                                prologue={"ops": ["log"]}, stream=0))
    assert st == 1
    st, _ = _status(lambda: hf.layout_convert(FAKE_IN, [3, 4], "f32", [1, 0], [1, 1], FAKE_OUT, stream=0))
    assert st == 1


def _q(scales, zps, qd=None, smin=-128, smax=127):
    return {"host_scales": np.array(scales, np.float32), "host_zero_points": np.array(zps, np.int32),
            "scales": 0x7000 if qd is not None else None, "zero_points": 0x8000 if qd is not None else None,
            "quantization_dimension": qd, "storage_min": smin, "storage_max": smax}


def test_quant_validation(lib):
    out_q = _q([0.05], [0])
    cases = [
        (_q([0.1, 0.2], [0, 0]), "C11"),                     # per-tensor with two scales
        (_q([0.1, 0.2, 0.3], [0, 0, 0], qd=1), "C13"),       # per-axis size mismatch
        (_q([0.0], [0]), "C6"),                              # scale must be > 0
        (_q([float("inf")], [0]), "C7"),                     # finite
        (_q([0.1], [200]), "C8"),                            # zero point in storage range
        (_q([0.1], [0], smin=5, smax=5), "C4"),              # storage_min < storage_max
        (_q([0.1], [0], qd=4), "C12"),                       # quantization_dimension in range
    ]
    for in_q, tag in cases:
        st, msg = _status(lambda: hf.quant_fusion(FAKE_IN, [4, 5], in_q, [0, 1], FAKE_OUT, out_q=out_q, stream=0))
        assert st == 1 and tag in msg, (tag, msg)
    # float output requires f32
    st, _ = _status(lambda: hf.quant_fusion(FAKE_IN, [4, 5], _q([0.1], [0]), [0, 1], FAKE_OUT, out_dtype="s8",
                                            out_q=None, stream=0))
    assert st == 1


def test_workspace_size_is_zero(lib):
    assert hf.reduce_workspace_size([8192, 16384], "bf16", [0]) == 0


def test_argmax_validation(lib):
    x, out = FAKE_IN, FAKE_OUT
    out_idx = FAKE_OUT + 4096
    # without an index input exactly one dimension is reduced
    st, msg = _status(lambda: hf.reduce_max_argmax(x, [4, 5], "f32", [0, 1], out, out_idx, stream=0))
    assert st == 1 and "one dimension" in msg
    # repeated dimension (C5) and out-of-range dimension (C4)
    idx = FAKE_IN + 8192
    st, msg = _status(lambda: hf.reduce_max_argmax(x, [4, 5], "f32", [1, 1], out, out_idx, indices=idx, stream=0))
    assert st == 1 and "C5" in msg
    st, msg = _status(lambda: hf.reduce_max_argmax(x, [4, 5], "f32", [3], out, out_idx, stream=0))
    assert st == 1 and "C4" in msg
    # integer values are not supported; the values output overlapping the input is rejected
    st, _ = _status(lambda: hf.reduce_max_argmax(x, [4, 5], "s32", [1], out, out_idx, stream=0))
    assert st == 2
    st, msg = _status(lambda: hf.reduce_max_argmax(x, [4, 5], "f32", [1], x + 8, out_idx, stream=0))
    assert st == 1 and "overlap" in msg
    # init_index outside s32
    st, msg = _status(lambda: hf.reduce_max_argmax(x, [4, 5], "f32", [1], out, out_idx, init_index=1 << 40, stream=0))
    assert st == 1 and "s32" in msg


# ---- constants of the correctly rounded f32 exp ------------------------------------------------------------
def test_exp_table_matches_its_generator(tmp_path):
    """exp_table.inc is what gen_exp_table.py writes (Python decimal, exact conversions)."""
    import importlib.util
    csrc = os.path.join(ROOT, "transpose_heroes_gb300", "csrc")
    spec = importlib.util.spec_from_file_location("gen_exp_table", os.path.join(csrc, "gen_exp_table.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    out = tmp_path / "exp_table.inc"
    gen.main(str(out))
    with open(os.path.join(csrc, "exp_table.inc")) as f:
        assert out.read_text() == f.read()


def test_exp_first_reduction_step_is_exact():
    """The f32 exp pass relies on r1 = x - k*L1f being exact (k = rint(64 x / ln2) from the f32 constant):
    check it on a million f32 arguments spread over the range and on the range ends."""
    import re
    with open(os.path.join(ROOT, "transpose_heroes_gb300", "csrc", "exp_table.inc")) as f:
        text = f.read()
    inv = float.fromhex(re.search(r"HLO_EXPF_INV64_LN2 (\S+)f", text).group(1))
    l1 = float.fromhex(re.search(r"HLO_EXPF_L1 (\S+)f", text).group(1))
    g = np.random.default_rng(5)
    x = np.concatenate([g.uniform(-87, 88.5, 1_000_000), [-87.0, 88.4999, 1e-30, -1e-30, 0.0054, -0.0054]])
    x = x.astype(np.float32).astype(np.float64)
    k = np.rint(x * np.float32(inv).astype(np.float64))  # x * INV is exact in f64; fma rounds it to an integer
    r1 = x - k * l1
    assert np.array_equal(r1.astype(np.float32).astype(np.float64), r1)
    assert np.abs(r1).max() < 0.04


def _expf_first_pass_emulated(x):
    """The f32 exp first pass of cr_exp.cuh, step for step in numpy (an FMA is emulated in f64: the
    product is exact there and the sum rounds once, twice only in rare ties, which a sampled bound
    tolerates). Returns (yh, yl, e) with exp(x) ~ (yh + yl) 2^e."""
    import re
    with open(os.path.join(ROOT, "transpose_heroes_gb300", "csrc", "exp_table.inc")) as f:
        text = f.read()
    c = {k: np.float32(float.fromhex(re.search(r"HLO_EXPF_%s (\S+)f" % k, text).group(1)))
         for k in ("INV64_LN2", "L1", "L2", "L3")}
    tab = re.findall(r"\{(\S+)f, (\S+)f\}", text.split("kExpTf")[1].split("};")[0])
    th = np.array([float.fromhex(a) for a, _ in tab], np.float32)
    tl = np.array([float.fromhex(b) for _, b in tab], np.float32)
    f32 = np.float32

    def fma(a, b, cc):
        return (np.asarray(a, np.float64) * np.asarray(b, np.float64) + np.asarray(cc, np.float64)).astype(f32)

    m = f32(12582912.0)
    t = fma(x, c["INV64_LN2"], m)
    k = t.view(np.int32) - 0x4B400000
    kf = (t - m).astype(f32)
    r1 = fma(-kf, c["L1"], x)
    p2h = (kf * c["L2"]).astype(f32)
    p2l = fma(kf, c["L2"], -p2h)
    rh = (r1 - p2h).astype(f32)
    bb = (rh - r1).astype(f32)
    rl = ((r1 - (rh - bb).astype(f32)).astype(f32) + (-p2h - bb).astype(f32)).astype(f32)
    rl = fma(-kf, c["L3"], (rl - p2l).astype(f32))
    q = fma(rh, f32(float.fromhex("0x1.555556p-5")), f32(float.fromhex("0x1.555556p-3")))
    q = fma(rh, q, f32(0.5))
    pe = fma((rh * rh).astype(f32), q, rl)
    pe = fma(rl, rh, pe)
    j = k & 63
    ah = (th[j] * rh).astype(f32)
    al = fma(th[j], rh, -ah)
    lo = fma(th[j], pe, tl[j])
    lo = (fma(tl[j], rh, lo) + al).astype(f32)
    yh = (th[j] + ah).astype(f32)
    yl = ((ah - (yh - th[j]).astype(f32)).astype(f32) + lo).astype(f32)
    return yh, yl, k >> 6


def test_expf_first_pass_error_below_its_rounding_bound():
    """The bound the kernel's rounding test uses (2^-35 on yh + yl, which lies in [1, 2.02)) holds with
    a margin: the emulated first pass stays within 2^-36.5 of exp(x) 2^-e (long double reference)."""
    g = np.random.default_rng(7)
    x = np.concatenate([g.uniform(-87, 88.5, 200_000), g.uniform(-0.01, 0.01, 50_000)]).astype(np.float32)
    yh, yl, e = _expf_first_pass_emulated(x)
    ref = np.exp(x.astype(np.longdouble)) / np.ldexp(np.longdouble(1), e)
    err = np.abs(yh.astype(np.longdouble) + yl.astype(np.longdouble) - ref)
    assert float(err.max()) < 2.0 ** -36.5


def test_logf_first_pass_error_below_its_rounding_bound():
    """The packed f32 log first pass (cr_log.cuh, cr_logf_first2 / cr_logf_first4), emulated step for step
    from the committed 32-interval tables: |log x - (S + lo)| stays below 2^-33.6 on U(0.5, 2), near 1,
    over the whole exponent range and on random normal bit patterns, so the test's bound b = 2^-33.5,
    less the rounding of lo +- b (< 2^-37), covers it. The same emulation over every positive normal
    float gives 2^-34.13 at most."""
    f32 = np.float32
    with open(os.path.join(ROOT, "transpose_heroes_gb300", "csrc", "log_table.inc")) as f:
        txt = f.read()

    def table(name):
        body = re.search(name + r"\[32\] = \{(.*?)\};", txt, re.S).group(1)
        return np.array([float.fromhex(v.strip().rstrip("f")) if v.strip() != "0.0f" else 0.0
                         for v in body.split(",") if v.strip()], dtype=f32)

    inv, hi, lo = table("kLog1Inv"), table("kLog1Hi"), table("kLog1Lo")
    off = int(re.search(r"HLO_LOG1_OFF (0x[0-9A-Fa-f]+)u", txt).group(1), 16)
    shift = int(re.search(r"HLO_LOG1_SHIFT (\d+)", txt).group(1))
    ln2a = f32(float.fromhex(re.search(r"HLO_LOG1_LN2_A (\S+)f", txt).group(1)))
    ln2b = f32(float.fromhex(re.search(r"HLO_LOG1_LN2_B (\S+)f", txt).group(1)))

    def fma(a, b, c):  # one rounding: the f64 product is exact, the sum's error is added back (TwoSum)
        p = np.asarray(a, np.float64) * np.asarray(b, np.float64)
        c = np.broadcast_to(np.asarray(c, np.float64), p.shape)
        s = p + c
        bb = s - p
        return (s + ((p - (s - bb)) + (c - bb))).astype(f32)

    g = np.random.default_rng(21)
    x = np.concatenate([g.uniform(0.5, 2.0, 1_500_000), 1.0 + g.uniform(-0.03, 0.03, 1_000_000),
                        np.exp(g.uniform(-87.0, 88.0, 1_000_000))]).astype(f32)
    x = np.concatenate([x, g.integers(0x00800000, 0x7F800000, 1_000_000, dtype=np.uint32).view(f32)])
    ix = x.view(np.uint32)
    t = (ix - np.uint32(off)).astype(np.uint32)
    i = (t >> np.uint32(shift)) & np.uint32(31)
    m = (ix - (t & np.uint32(0xFF800000))).astype(np.uint32).view(f32)
    e = (t.view(np.int32) >> 23).astype(f32)
    r = fma(m, inv[i], f32(-1))
    a = fma(e, ln2a, hi[i])
    s = (a + r).astype(f32)
    err_sum = (r - (s - a).astype(f32)).astype(f32)
    p = fma(r, f32(0.2), f32(-0.25))
    p = fma(r, p, f32(0.33333334))
    p = fma(r, p, f32(-0.5))
    b = fma(e, ln2b, lo[i])
    rest = fma((r * r).astype(f32), p, b)
    lo_ = (err_sum + rest).astype(f32)
    err = np.abs(s.astype(np.float64) + lo_.astype(np.float64) - np.log(x.astype(np.float64)))
    assert float(err.max()) < 2.0 ** -33.6


def test_tanhf_first_pass_errors_below_their_rounding_bounds():
    """Both branches of the f32 tanh first pass (cr_exp.cuh), emulated step for step: the Taylor branch
    (a < 2^-4) within 2^-39 a of tanh a (the test uses a 2^-37), the 1 - 2/(exp(2a) + 1) branch within
    2^-37.5 absolute (the test uses 2^-35.5)."""
    f32 = np.float32

    def fma(a, b, c):
        return (np.asarray(a, np.float64) * np.asarray(b, np.float64) + np.asarray(c, np.float64)).astype(f32)

    h = lambda s: f32(float.fromhex(s))
    g = np.random.default_rng(8)
    a = np.concatenate([g.uniform(2.0 ** -20, 0.0625, 100_000), np.geomspace(1e-30, 0.0624, 20_000)]).astype(f32)
    a = a[a < f32(0.0625)]
    a2h = (a * a).astype(f32)
    a2l = fma(a, a, -a2h)
    a3h = (a * a2h).astype(f32)
    a3l = fma(a, a2l, fma(a, a2h, -a3h))
    ch = (a3h * h("0x1.555556p-2")).astype(f32)
    cl = fma(a3l, h("0x1.555556p-2"), fma(a3h, h("-0x1.555556p-27"), fma(a3h, h("0x1.555556p-2"), -ch)))
    p = fma(a2h, h("-0x1.226e36p-7"), h("0x1.664f48p-6"))
    p = fma(a2h, p, h("-0x1.ba1ba2p-5"))
    p = fma(a2h, p, h("0x1.111112p-3"))
    t5 = ((a3h * a2h).astype(f32) * p).astype(f32)
    th = (a - ch).astype(f32)
    tl = (((a - th).astype(f32) - ch).astype(f32) + (t5 - cl).astype(f32)).astype(f32)
    err = np.abs(th.astype(np.longdouble) + tl.astype(np.longdouble) - np.tanh(a.astype(np.longdouble)))
    assert float((err / a.astype(np.longdouble)).max()) < 2.0 ** -39

    a = g.uniform(0.0625, 9.05, 200_000).astype(f32)
    yh, yl, e = _expf_first_pass_emulated((2 * a).astype(f32))
    sc = np.ldexp(f32(1), e).astype(f32)
    eh, el = (yh * sc).astype(f32), (yl * sc).astype(f32)
    d1 = (eh + f32(1)).astype(f32)
    d2 = ((f32(1) - (d1 - eh).astype(f32)).astype(f32) + el).astype(f32)
    dh = (d1 + d2).astype(f32)
    dl = (d2 - (dh - d1).astype(f32)).astype(f32)
    q0 = (f32(2) / dh).astype(f32)
    r = fma(-q0, dl, fma(-q0, dh, f32(2)))
    q1 = (r * (q0 * f32(0.5)).astype(f32)).astype(f32)
    th = (f32(1) - q0).astype(f32)
    tl = (((f32(1) - th).astype(f32) - q0).astype(f32) - q1).astype(f32)
    err = np.abs(th.astype(np.longdouble) + tl.astype(np.longdouble) - np.tanh(a.astype(np.longdouble)))
    assert float(err.max()) < 2.0 ** -37.5


def test_quantized_data_movement_validation(lib):
    """broadcast_in_dim C3-C5 and reshape C1-C3 are checked before anything is enqueued."""
    # per-axis operands need device parameter pointers: fake ones, never dereferenced
    q = {"scales": 0x300000, "zero_points": 0x310000, "host_scales": np.float32([0.2, 0.1, 0.3]),
         "host_zero_points": np.int32([20, 10, 30]), "quantization_dimension": 1}
    sc, zp = FAKE_OUT + (1 << 20), FAKE_OUT + (2 << 20)
    # C3: broadcast dimension out of range; C4: repeated; C5: size mismatch
    for bdims, out_dims, tag in [([0, 3], [2, 3, 2], "C3"), ([2, 2], [2, 3, 2], "C4"), ([0, 2], [2, 3, 4], "C5")]:
        st, msg = _status(lambda: hf.quant_broadcast_in_dim(FAKE_IN, [2, 3], q, bdims, FAKE_OUT, out_dims, sc, zp,
                                                            stream=0))
        assert st == 1 and tag in msg, msg
    # reshape C2 (element count), C3 (quantized axis kept), C1 (per-tensor stays per-tensor)
    st, msg = _status(lambda: hf.reshape(FAKE_IN, [4, 3, 2], FAKE_OUT, [5, 5], "s8", q=None, stream=0))
    assert st == 1 and "C2" in msg
    q3 = q
    for out_dims, rqd in [([12, 2], 0), ([4, 6], 1), ([2, 2, 3, 2], 1)]:
        st, msg = _status(lambda: hf.reshape(FAKE_IN, [4, 3, 2], FAKE_OUT, out_dims, "s8", q=q3, result_qdim=rqd,
                                             stream=0))
        assert st == 1 and "C3" in msg, msg
    pt = {"host_scales": np.float32([0.1]), "host_zero_points": np.int32([0]), "quantization_dimension": None}
    st, msg = _status(lambda: hf.reshape(FAKE_IN, [4, 3, 2], FAKE_OUT, [24], "s8", q=pt, result_qdim=0, stream=0))
    assert st == 1 and "C1" in msg


def test_reduce_workspace_rules(lib):
    """Few long rows ask for a workspace (one f32 partial per row segment); a non-NULL workspace that is
    too small is HLO_ERR_WORKSPACE; many rows, or a column reduce, need none."""
    need = hf.reduce_workspace_size([1, 1 << 24], "f32", [1])
    assert need > 0 and need % 4 == 0
    assert hf.reduce_workspace_size([4096, 4096], "f32", [1]) == 0
    assert hf.reduce_workspace_size([1 << 20, 8], "f32", [0]) == 0
    big_in, big_out, ws = 1 << 32, 1 << 34, 1 << 36  # never dereferenced, and far apart
    st, msg = _status(lambda: hf.reduce_fusion(big_in, [1, 1 << 24], "f32", [1], "add", 0.0, big_out, "f32",
                                               workspace=ws, workspace_bytes=4, stream=0))
    assert st == 4 and "workspace" in msg


def test_tanh_table_matches_its_generator(tmp_path):
    """tanh_table.inc is what gen_tanh_table.py writes (Python decimal, exact bf16 rounding)."""
    import importlib.util
    csrc = os.path.join(ROOT, "transpose_heroes_gb300", "csrc")
    spec = importlib.util.spec_from_file_location("gen_tanh_table", os.path.join(csrc, "gen_tanh_table.py"))
    gen = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(gen)
    out = tmp_path / "tanh_table.inc"
    gen.main(str(out))
    with open(os.path.join(csrc, "tanh_table.inc")) as f:
        assert out.read_text() == f.read()


def test_tanh_table_against_the_oracle():
    """Every entry of the bf16 tanh table equals the oracle's correctly rounded bf16 tanh of that
    argument, for both signs (the kernel copies the sign of x onto the entry of |x|)."""
    import re
    with open(os.path.join(ROOT, "transpose_heroes_gb300", "csrc", "tanh_table.inc")) as f:
        tab = np.array([int(v, 16) for v in re.findall(r"0x([0-9A-F]{4})", f.read())], dtype=np.uint32)
    assert len(tab) == 32768
    import oracle
    data = np.arange(1 << 16, dtype=np.uint16)
    ref = oracle.transpose(data, [1 << 16], "bf16", [0], prologue={"ops": ["tanh"], "round_each": True})
    ref = ref.view(np.uint16).astype(np.uint32)
    got = tab[data & 0x7FFF] | (data.astype(np.uint32) & 0x8000)
    bf = lambda b: (b.astype(np.uint32) << 16).view(np.float32)
    same = (got == ref) | (np.isnan(bf(got)) & np.isnan(bf(ref)))
    assert same.all(), np.flatnonzero(~same)[:8]


# ---- host-side fault injection (HLOFUSION_FAULT) -----------------------------------------------------------
def _valid_calls():
    """One valid call per entry point that enqueues work; the pointers are never dereferenced because
    the injected fault returns before anything is launched."""
    q = {"scales": np.float32([0.5]), "zero_points": np.int32([0]), "quantization_dimension": None,
         "host_scales": np.float32([0.5]), "host_zero_points": np.int32([0]), "storage_min": -128, "storage_max": 127}
    return {
        "hlo_reduce_fusion": lambda: hf.reduce_fusion(FAKE_IN, [4, 5], "f32", [1], "add", 0.0, FAKE_OUT, "f32", stream=0),
        "hlo_transpose_fusion": lambda: hf.transpose_fusion(FAKE_IN, [3, 4], "f32", [1, 0], FAKE_OUT, stream=0),
        "hlo_layout_convert": lambda: hf.layout_convert(FAKE_IN, [3, 4], "f32", [1, 0], [0, 1], FAKE_OUT, stream=0),
        "hlo_quant_binary": lambda: hf.quant_binary("add", FAKE_IN, FAKE_IN + 4096, [64], q, q, FAKE_OUT, q, stream=0),
    }


@pytest.mark.parametrize("site", ["hlo_reduce_fusion", "hlo_transpose_fusion", "hlo_layout_convert", "hlo_quant_binary"])
def test_fault_injection_by_entry_point(lib, monkeypatch, site):
    """HLOFUSION_FAULT=<entry point> makes that call return HLO_ERR_CUDA ("injected fault") after
    validation and before any launch; an invalid call still reports its own validation error."""
    calls = _valid_calls()
    monkeypatch.setenv("HLOFUSION_FAULT", site)
    st, msg = _status(calls[site])
    assert st == 3 and "injected fault" in msg and site in msg
    if site == "hlo_transpose_fusion":
        st, msg = _status(lambda: hf.transpose_fusion(FAKE_IN, [3, 4], "f32", [0, 0], FAKE_OUT, stream=0))
        assert st == 1 and "permutation" in msg
    monkeypatch.setenv("HLOFUSION_FAULT", "all")
    for name, call in calls.items():
        st, msg = _status(call)
        assert st == 3 and "injected fault" in msg and name in msg


def test_fault_injection_names_one_site(lib, monkeypatch):
    """A site names one entry point: with HLOFUSION_FAULT set to another, the call goes on past the
    injection point (here, on a host without a GPU, to the CUDA runtime's own error)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("the call would really launch on a GPU host")
    monkeypatch.setenv("HLOFUSION_FAULT", "hlo_reduce_fusion")
    st, msg = _status(_valid_calls()["hlo_transpose_fusion"])
    assert "injected fault" not in msg


# ---- the run-time chain generator (jit_chain.cu), through hlo_jit_source: no device needed ------------------
GELU = {"ops": ["mul_input", "mul_input", ("mul_const", 0.044708), "add_input", ("mul_const", 0.79785), "tanh",
                ("add_const", 1.0), ("mul_const", 0.5), "mul_input"], "round_each": True}
TWO_TANH_RUNS = {"ops": ["mul_input", "tanh", "add_input", "tanh", ("mul_const", 2.0), "mul_input"], "round_each": True}
NO_TANH_F16 = {"ops": ["mul_input", ("add_const", -1.5), "neg", ("mul_const", 0.3), "add_input", "abs"],
               "round_each": True}


def _defines(src):
    return dict(re.findall(r"^#define (\w+) (\S+)$", src, re.M))


def _chain_function(src):
    return re.search(r"u32 f\(u32 x, const unsigned short\* t\) \{(.*?)\n\}", src, re.S).group(1)


def test_jit_source_table_plans(lib):
    """GELU's tanh sits in one x-free run of four ops (multiply, tanh, add 1, multiply): one 65536-entry
    run table (128 KiB, six ring stages) and a table-building kernel that applies exactly those ops; a
    chain with tanh in two runs reads the 64 KiB tanh table; a chain without tanh has no table."""
    src = hf.jit_source(GELU, "bf16")
    d = _defines(src)
    assert (d["TB"], d["NS"], d["CB"]) == ("131072", "6", "16384")
    body = _chain_function(src)
    assert body.count("hmul(v, x)") == 3 and body.count("hadd(v, x)") == 1
    assert "hlook(v, t)" in body and "htanh" not in body
    table = re.search(r"hlo_jit_table\(.*?\{(.*?)\n\}", src, re.S).group(1)
    run = re.findall(r"v = (\w+)\(v, (0x[0-9A-F]+u|t)\)", table)
    # bf16 bits: 0.79785 -> 0x3F4C, 1 -> 0x3F80, 0.5 -> 0x3F00, each in both halves of the pair
    assert run == [("hmul", "0x3F4C3F4Cu"), ("htanh", "t"), ("hadd", "0x3F803F80u"), ("hmul", "0x3F003F00u")]

    src = hf.jit_source(TWO_TANH_RUNS, "bf16")
    assert _defines(src)["TB"] == "65536" and "hlo_jit_table" not in src
    assert _chain_function(src).count("htanh(v, t)") == 2

    src = hf.jit_source(NO_TANH_F16, "f16")
    d = _defines(src)
    assert d["TB"] == "0" and d["NS"] == "12" and "add.rn.f16x2" in src and "bf16" not in src
    assert "v ^= 0x80008000u" in src and "v &= 0x7FFF7FFFu" in src


def test_jit_source_rejects_other_chains(lib):
    """The generator takes rounded 16-bit chains of adds, multiplies, negate, abs and bf16 tanh only."""
    assert hf.jit_source({"ops": ["exp"], "round_each": True}, "bf16") is None
    assert hf.jit_source({"ops": ["tanh"], "round_each": True}, "f16") is None
    assert hf.jit_source({"ops": ["abs"], "round_each": False}, "bf16") is None
    assert hf.jit_source({"ops": ["abs"], "round_each": True}, "f32") is None
    assert hf.jit_source({"ops": ["abs"], "round_each": True}, "bf16") is not None
    chain = hf.make_chain({"ops": ["abs"], "round_each": True})
    assert lib.hlo_jit_source(ctypes.byref(chain), hf.DTYPES["bf16"], None, 5) == -1  # NULL buffer, length 5
    n = lib.hlo_jit_source(ctypes.byref(chain), hf.DTYPES["bf16"], None, 0)
    small = ctypes.create_string_buffer(8)
    assert lib.hlo_jit_source(ctypes.byref(chain), hf.DTYPES["bf16"], small, 8) == n and small.value == b""


@pytest.mark.parametrize("spec,dtype", [(GELU, "bf16"), (TWO_TANH_RUNS, "bf16"), (NO_TANH_F16, "f16")])
def test_jit_source_compiles_for_sm_103a(lib, spec, dtype, tmp_path):
    """The generated source compiles for sm_103a (nvcc here stands in for NVRTC on the device), with no
    register spills."""
    import shutil
    import subprocess

    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    src = tmp_path / "chain.cu"
    src.write_text(hf.jit_source(spec, dtype))
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-Xptxas", "-v", "-c",
                        str(src), "-o", str(tmp_path / "chain.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    assert " 0 bytes spill stores" in r.stderr and "bytes spill stores" in r.stderr
    assert all(m == "0" for m in re.findall(r"(\d+) bytes spill stores", r.stderr))
