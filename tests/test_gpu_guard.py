"""Guard bands around every output: each kernel family writes into a buffer with 4 KiB of a known byte
pattern on both sides, on ragged and unaligned sizes, and the pattern must be untouched afterwards
(a stray write past either end of an output fails here even where the parity tests would pass). The
outputs themselves are checked against the oracle as in the parity tests.
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import transpose_heroes_gb300 as hf
from transpose_heroes_gb300 import inputs as inp
from transpose_heroes_gb300.runner import DeviceFusion

from test_gpu_parity import check, run_oracle

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transpose_heroes_gb300 import build

    build.build()
    oracle.build()
    hf.lib()


class Guarded:
    """nbytes of output with GUARD bytes of PATTERN before and after; `shift` extra bytes in front make the
    output start off a 16-byte boundary."""

    def __init__(self, nbytes, shift=0):
        self.raw = torch.full((nbytes + 2 * GUARD + shift,), PATTERN, dtype=torch.uint8, device="cuda")
        self.lo = GUARD + shift
        self.nbytes = nbytes

    def view(self, dtype):
        return self.raw[self.lo:self.lo + self.nbytes].view(dtype)

    def assert_intact(self, what=""):
        r = self.raw.cpu().numpy()
        before, after = r[:self.lo], r[self.lo + self.nbytes:]
        bad_b, bad_a = np.flatnonzero(before != PATTERN), np.flatnonzero(after != PATTERN)
        assert bad_b.size == 0, f"{what}: {bad_b.size} guard bytes before the output overwritten (first at -{self.lo - bad_b[0]})"
        assert bad_a.size == 0, f"{what}: {bad_a.size} guard bytes after the output overwritten (first at +{bad_a[0]})"


def run_guarded(f, shift=0):
    d = DeviceFusion(f)
    g = Guarded(d.out.numel() * d.out.element_size(), shift)
    d.out = g.view(d.out.dtype)
    d.run()
    torch.cuda.synchronize()
    g.assert_intact(f.name)
    return d.output_numpy()


def _reduce(name, data, dims, dtype, dimensions, kind, ops=None, init=0.0, out_dtype="f32", m2m=None):
    m2m = m2m or list(range(len(dims) - 1, -1, -1))
    kept = [dims[d] for d in range(len(dims)) if d not in dimensions]
    return inp.Fusion(name=name, kind="reduce", dims=dims, m2m=m2m, dtype=dtype, data=data, dimensions=dimensions,
                      reduce_kind=kind, init=init, prologue={"ops": ops, "round_each": True} if ops else None,
                      out_dims=kept, out_m2m=list(range(len(kept) - 1, -1, -1)), out_dtype=out_dtype)


def _transpose(name, data, dims, dtype, perm, pro=None, epi=None, self_add=False, m2m=None, out_m2m=None):
    m2m = m2m or list(range(len(dims) - 1, -1, -1))
    out_dims = [dims[p] for p in perm]
    return inp.Fusion(name=name, kind="transpose", dims=dims, m2m=m2m, dtype=dtype, data=data, permutation=perm,
                      self_add=self_add, prologue=pro, epilogue=epi, out_dims=out_dims,
                      out_m2m=out_m2m or list(range(len(dims) - 1, -1, -1)), out_dtype=dtype)


def _cases():
    g = inp.rng(77)
    f32 = lambda n, lo=-1.0, hi=1.0: inp.uniform_f32(g, n, lo, hi)  # noqa: E731
    cases = {
        "row_reduce_vec": inp.row_reduce_exp(seed=3, rows=37, cols=1000),
        "row_reduce_scalar": inp.row_reduce_exp(seed=3, rows=5, cols=1001),
        "row_stream": inp.bcast_exp_reduce(seed=3, d0=1, d2=70, d3=8200),
        "row_reduce_rt": _reduce("rt", f32(33 * 77), [33, 77], "f32", [1], "add", ["neg", "exp"]),
        "col_reduce_vec": inp.col_reduce_max(seed=3, rows=301, cols=1024),
        "col_reduce_scalar": inp.col_reduce_max(seed=3, rows=301, cols=1030),
        "gen_reduce": _reduce("gen", f32(120), [4, 5, 6], "f32", [0, 2], "add", ["exp"]),
        "fill": _reduce("fill", np.zeros(0, np.float32), [3, 0], "f32", [1], "max", init=2.5),
        "selfadd_tma": inp.transpose_log(seed=3, n=130),
        "selfadd_pair": inp.transpose_log(seed=3, n=131),
        "tile_transpose": inp.transpose3_exp_abs(seed=3, dims=(20, 160, 170)),
        "gather_bcast": _transpose("gb", f32(42), [6, 7], "f32", [1, 0],
                                   pro={"ops": ["add_bcast"], "bcast": {"data": f32(7), "dims": [7], "dtype": "f32",
                                                                        "broadcast_dimensions": [1]}}),
        "elementwise_f32": _transpose("ew", f32(1003), [1003], "f32", [0], pro={"ops": ["tanh"], "round_each": True}),
        "elementwise_16x2": inp.gelu_bf16(seed=3, dims=(3, 7, 1001)),
        # a bf16 chain with exp from 2^22 elements: the chain's table kernel (the generated kernels do
        # not take exp)
        "elementwise_lut16": _transpose("lut", inp.normal_bf16(g, (1 << 22) + 7), [(1 << 22) + 7], "bf16", [0],
                                        pro={"ops": ["exp", ("mul_const", 0.5)], "round_each": True}),
        # the generated kernels (from 2^20 elements, 16-byte aligned): GELU with its run table and a
        # partial last chunk per block plus a 5-element tail; an f16 chain with no table
        "generated_run_table": inp.gelu_bf16(seed=3, dims=(64, 256, 257)),
        "generated_tail": inp.gelu_bf16(seed=3, dims=((1 << 20) + 5,)),
        "generated_no_table": _transpose("gen_f16", (inp.uniform_f32(g, (1 << 21) + 3, -4.0, 4.0)
                                                     .astype(np.float16).view(np.uint16)), [(1 << 21) + 3], "f16", [0],
                                         pro={"ops": ["mul_input", ("add_const", -1.5), "abs"], "round_each": True}),
        "copy": _transpose("copy", f32(999), [999], "f32", [0]),
        "quant_tile_ragged": inp.quant_relayout(seed=3, n0=301, n1=517),
        "quant_tile_full": inp.quant_relayout(seed=3, n0=256, n1=384),
    }
    qf = inp.quant_relayout(seed=4, n0=33, n1=65)
    qf.out_q, qf.out_dtype, qf.name = None, "f32", "quant_gather_f32"
    cases["quant_gather_f32"] = qf
    return cases


CASES = _cases()


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("shift", [0, 4])
def test_fusion_outputs_stay_in_bounds(name, shift):
    f = CASES[name]
    ref, asum = run_oracle(f)
    check(f, run_guarded(f, shift), ref, asum)


@pytest.mark.parametrize("shape,dims", [([37, 1000], [1]), ([6, 50, 33], [0, 2])])
def test_argmax_outputs_stay_in_bounds(shape, dims):
    g = np.random.default_rng(9)
    n = int(np.prod(shape))
    x = g.standard_normal(n).astype(np.float32)
    k = g.permutation(n).astype(np.int32) if len(dims) > 1 else None
    ref_v, ref_i = oracle.reduce_max_argmax(x, shape, "f32", dims, -math.inf, -1, indices=k)
    n_out = ref_v.size
    gv, gi = Guarded(4 * n_out), Guarded(4 * n_out)
    hf.reduce_max_argmax(torch.from_numpy(x).cuda(), shape, "f32", dims, gv.view(torch.float32), gi.view(torch.int32),
                         indices=torch.from_numpy(k).cuda() if k is not None else None)
    torch.cuda.synchronize()
    gv.assert_intact("argmax values")
    gi.assert_intact("argmax indices")
    assert np.array_equal(gv.view(torch.float32).cpu().numpy(), ref_v)
    assert np.array_equal(gi.view(torch.int32).cpu().numpy(), ref_i)


def _qpt(scale, zp):
    return {"host_scales": np.float32([scale]), "host_zero_points": np.int32([zp]), "quantization_dimension": None}


@pytest.mark.parametrize("n,shift", [(4099, 0), (4099, 1), ((1 << 22) + 5, 0)])
def test_quant_binary_outputs_stay_in_bounds(n, shift):
    """The vector kernel (aligned), the per-element kernel (shifted) and the pair-table kernel (2^22+)."""
    g = np.random.default_rng(n)
    a = g.integers(-128, 128, n).astype(np.int8)
    b = g.integers(-128, 128, n).astype(np.int8)
    ql, qr, qo = _qpt(0.0371, 4), _qpt(0.113, -9), _qpt(0.09, 2)
    ref = oracle.quant_binary("add", a, b, [n], dict(scales=[0.0371], zero_points=[4]),
                              dict(scales=[0.113], zero_points=[-9]), dict(scales=[0.09], zero_points=[2]))
    out = Guarded(n, shift)
    hf.quant_binary("add", torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), [n], ql, qr, out.view(torch.int8), qo)
    torch.cuda.synchronize()
    out.assert_intact("quantized add")
    assert np.array_equal(out.view(torch.int8).cpu().numpy(), ref)


def test_quant_data_movement_outputs_stay_in_bounds():
    g = np.random.default_rng(8)
    dims, out_dims = [5, 1, 7], [5, 3, 7, 2]
    q = {"scales": g.uniform(0.01, 0.5, 7).astype(np.float32), "zero_points": g.integers(-20, 21, 7).astype(np.int32),
         "quantization_dimension": 2}
    codes = g.integers(-128, 128, size=dims).astype(np.int8)
    ref, params = oracle.quant_broadcast_in_dim(codes.ravel(), dims, q, [0, 1, 2], out_dims)
    n_out = int(np.prod(out_dims))
    out, rs, rz = Guarded(n_out, 3), Guarded(4 * 7), Guarded(4 * 7)
    dq = {"scales": torch.from_numpy(q["scales"]).cuda(), "zero_points": torch.from_numpy(q["zero_points"]).cuda(),
          "host_scales": q["scales"], "host_zero_points": q["zero_points"], "quantization_dimension": 2}
    rqd = hf.quant_broadcast_in_dim(torch.from_numpy(codes.ravel()).cuda(), dims, dq, [0, 1, 2], out.view(torch.int8),
                                    out_dims, rs.view(torch.float32), rz.view(torch.int32))
    torch.cuda.synchronize()
    for gd, what in ((out, "codes"), (rs, "scales"), (rz, "zero points")):
        gd.assert_intact("quantized broadcast_in_dim " + what)
    assert rqd == 2 and np.array_equal(out.view(torch.int8).cpu().numpy(), ref)
    assert np.array_equal(rs.view(torch.float32).cpu().numpy(), params["scales"])
    # reshape with layouts (the gather kernel)
    x = g.integers(-1000, 1000, size=[9, 10, 11]).astype(np.int32)
    ref = oracle.reshape(x.ravel(), [9, 10, 11], [11, 90], "s32", out_m2m=[0, 1])
    out = Guarded(4 * x.size, 4)
    hf.reshape(torch.from_numpy(x.ravel()).cuda(), [9, 10, 11], out.view(torch.int32), [11, 90], "s32", out_m2m=[0, 1])
    torch.cuda.synchronize()
    out.assert_intact("reshape")
    assert np.array_equal(out.view(torch.int32).cpu().numpy(), ref)
