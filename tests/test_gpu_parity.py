"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the same seeded inputs.

Bars (from the fusion semantics):
  * transposes, layout changes and quantized relayouts: bit-exact (log is correctly rounded in f32);
  * float reductions with add: |gpu - oracle| <= 1e-5 * sum|terms| + 1e-6 (f32 accumulation against the
    oracle's long-double sum), plus half an output ulp when the output type is 16-bit;
  * reductions with max: bit-exact.
Sizes: scaled-down shapes that span several tiles and end in ragged tails, the full-size workloads in
the launch configuration the benchmark times, and edge cases (empty, unit and unaligned).
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import transpose_heroes_gb300 as hf
from transpose_heroes_gb300 import inputs as inp
from transpose_heroes_gb300.runner import DeviceFusion

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transpose_heroes_gb300 import build

    build.build()
    oracle.build()
    hf.lib()


def run_gpu(f):
    d = DeviceFusion(f)
    d.run()
    torch.cuda.synchronize()
    return d.output_numpy()


def run_oracle(f):
    if f.kind == "reduce":
        return oracle.reduce(f.data, f.dims, f.dtype, f.dimensions, f.reduce_kind, f.init, f.out_dtype, m2m=f.m2m,
                             out_m2m=f.out_m2m, prologue=f.prologue, want_abs_sum=True)
    if f.kind == "transpose":
        return oracle.transpose(f.data, f.dims, f.dtype, f.permutation, m2m=f.m2m, out_m2m=f.out_m2m,
                                self_add=f.self_add, prologue=f.prologue, epilogue=f.epilogue), None
    if f.kind == "layout":
        return oracle.layout_convert(f.data, f.dims, f.dtype, f.m2m, f.out_m2m), None
    if f.kind == "quant":
        return oracle.quant_fusion(f.data, f.dims, f.dtype, f.in_q, f.out_m2m, f.out_dtype, out_q=f.out_q,
                                   m2m=f.m2m, float_ops=f.prologue), None
    raise ValueError(f.kind)


def as_f32(buf, dtype):
    if dtype in ("bf16",):
        return inp.bf16_bits_to_f32(buf)
    if dtype == "f16":
        return np.asarray(buf, np.uint16).view(np.float16).astype(np.float32)
    return np.asarray(buf, np.float32)


def check(f, gpu, ref, asum):
    assert gpu.shape == ref.shape
    if f.kind == "reduce" and f.reduce_kind == "add":
        g = as_f32(gpu, f.out_dtype).astype(np.float64)
        r = as_f32(ref, f.out_dtype).astype(np.float64)
        tol = 1e-5 * asum + 1e-6
        if f.out_dtype in ("bf16", "f16"):
            tol = tol + np.abs(r) * (2.0 ** -8 if f.out_dtype == "bf16" else 2.0 ** -11)
        err = np.abs(g - r)
        bad = ~(err <= tol)
        assert not bad.any(), f"{bad.sum()} outputs out of tolerance; worst err {err.max()} tol {tol[np.argmax(err)]}"
    else:
        if f.out_dtype in ("f32",):
            g, r = gpu.view(np.uint32), ref.view(np.uint32)
            nan_g, nan_r = np.isnan(gpu), np.isnan(ref)
            assert np.array_equal(nan_g, nan_r)
            same = (g == r) | nan_g
        elif f.out_dtype in ("bf16", "f16"):
            gf, rf = as_f32(gpu, f.out_dtype), as_f32(ref, f.out_dtype)
            same = (gpu.view(np.uint16) == ref.view(np.uint16)) | (np.isnan(gf) & np.isnan(rf))
        else:
            same = gpu == ref
        nbad = int((~same).sum())
        if nbad:
            where = np.flatnonzero(~same)[:4]
            detail = [(int(w), gpu.flat[w].item(), ref.flat[w].item()) for w in where]
            raise AssertionError(f"{nbad} of {same.size} outputs differ; (index, gpu, oracle): {detail}")


NAMES = list(inp.FULL)


@pytest.mark.parametrize("name", NAMES)
@pytest.mark.parametrize("seed", [1, 2])
def test_small_configs(name, seed):
    f = inp.small(name, seed=seed)
    ref, asum = run_oracle(f)
    check(f, run_gpu(f), ref, asum)


@pytest.mark.parametrize("name", NAMES)
def test_full_size_configs(name):
    """The full-size workloads, as the benchmark launches them, against the oracle on every output."""
    f = inp.full(name, seed=1)
    ref, asum = run_oracle(f)
    gpu = run_gpu(f)
    check(f, gpu, ref, asum)
    if name == "transpose_log":
        n = f.dims[0]
        g = gpu.view(np.uint32).reshape(n, n)
        assert np.array_equal(g, g.T)  # bitwise symmetric
    assert oracle.unresolved_count() == 0


def test_full_size_step_on_concurrent_streams():
    """The benchmark's step: the five full-size fusions each on a stream of its own (runner.
    ConcurrentFusions), twice in a row with the outputs cleared between, every output against the
    oracle; work queued on the caller's stream after the step sees all five outputs."""
    from transpose_heroes_gb300.runner import ConcurrentFusions

    fusions = [inp.full(n, seed=2) for n in NAMES]
    devs = [DeviceFusion(f) for f in fusions]
    torch.cuda.synchronize()
    step = ConcurrentFusions(devs)
    refs = [run_oracle(f) for f in fusions]
    stream = torch.cuda.current_stream()
    for _ in range(2):
        for d in devs:
            d.out.fill_(-1)
        step.run(stream)
        host = [torch.empty(d.out.shape, dtype=d.out.dtype, pin_memory=True) for d in devs]
        for h, d in zip(host, devs):
            h.copy_(d.out, non_blocking=True)  # on the caller's stream, after the join
        stream.synchronize()
        view = {"f32": np.float32, "bf16": np.uint16, "f16": np.uint16, "s8": np.int8}
        for f, h, (ref, asum) in zip(fusions, host, refs):
            check(f, h.numpy().view(view[f.out_dtype]), ref, asum)


def test_selfadd_beyond_2_to_31_elements():
    """The self-add transpose on f32[46404, 46404]: 2.15e9 elements, past every 32-bit element count and
    byte offset, with a ragged last tile row and column. 6144 sampled outputs (a third of them in the
    ragged tiles) against the oracle's correctly rounded logs, and bitwise symmetry on them."""
    n = 46404
    g = inp.rng(77)
    x = torch.empty(n * n, dtype=torch.float32, device="cuda")
    chunk = 1 << 26
    for s in range(0, n * n, chunk):
        m = min(chunk, n * n - s)
        x[s:s + m].copy_(torch.from_numpy(inp.uniform_f32(g, m, 0.5, 2.0)))
    y = torch.empty_like(x)
    hf.transpose_fusion(x, [n, n], "f32", [1, 0], y, self_add=True, prologue={"ops": ["log"]})
    torch.cuda.synchronize()
    rs = np.random.default_rng(78)
    i = np.concatenate([rs.integers(0, n, 4096), rs.integers(n - 70, n, 1024), rs.integers(0, n, 1024)])
    j = np.concatenate([rs.integers(0, n, 4096), rs.integers(0, n, 1024), rs.integers(n - 70, n, 1024)])
    ij = torch.from_numpy(i * n + j).cuda()
    ji = torch.from_numpy(j * n + i).cuda()
    pij, pji = x[ij].cpu().numpy(), x[ji].cpu().numpy()
    out_ij, out_ji = y[ij].cpu().numpy(), y[ji].cpu().numpy()
    ref = np.array([np.float32(oracle.log(a, "f32")) + np.float32(oracle.log(b, "f32")) for a, b in zip(pij, pji)],
                   dtype=np.float32)
    assert np.array_equal(out_ij.view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(out_ij.view(np.uint32), out_ji.view(np.uint32))
    del x, y
    torch.cuda.empty_cache()


def _fill_device(n, make, dtype):
    """A device buffer of n elements filled chunk by chunk from a host generator."""
    x = torch.empty(n, dtype=dtype, device="cuda")
    chunk = 1 << 26
    for s in range(0, n, chunk):
        m = min(chunk, n - s)
        x[s:s + m].copy_(torch.from_numpy(make(m)))
    return x


def test_col_reduce_beyond_2_to_31_elements():
    """Column reduce-max over bf16[65540, 32768] (2.15e9 elements): 64 sampled columns, the last ones
    among them, against the oracle on the same columns."""
    rows, cols = 65540, 32768
    g = inp.rng(79)
    x = _fill_device(rows * cols, lambda m: inp.normal_bf16(g, m).view(np.int16), torch.int16)
    out = torch.empty(cols, dtype=torch.int16, device="cuda")
    hf.reduce_fusion(x, [rows, cols], "bf16", [0], "max", float("-inf"), out, "bf16")
    torch.cuda.synchronize()
    cs = np.concatenate([np.random.default_rng(80).integers(0, cols, 56), np.arange(cols - 8, cols)])
    sub = x.view(rows, cols)[:, torch.from_numpy(cs).cuda()].contiguous().cpu().numpy().view(np.uint16)
    ref = oracle.reduce(sub.reshape(-1), [rows, len(cs)], "bf16", [0], "max", float("-inf"), "bf16")
    assert np.array_equal(out.cpu().numpy().view(np.uint16)[cs], ref.view(np.uint16))
    del x
    torch.cuda.empty_cache()


def test_quant_relayout_beyond_2_to_31_elements():
    """Per-axis dequantize -> {0,1} -> quantize on s8[46464, 46464] (2.16e9 codes, tensor-copy tiles):
    4096 sampled codes against the oracle's per-element dequantize and quantize."""
    n = 46464
    g = inp.rng(81)
    x = _fill_device(n * n, lambda m: inp.integers(g, m, -128, 127, np.int8), torch.int8)
    scales = inp.uniform_f32(g, n, 0.001, 0.1)
    zps = inp.integers(g, n, -20, 20, np.int32)
    qin = {"scales": torch.from_numpy(scales).cuda(), "zero_points": torch.from_numpy(zps).cuda(),
           "host_scales": scales, "host_zero_points": zps, "quantization_dimension": 1,
           "storage_min": -128, "storage_max": 127}
    qout = {"scales": np.float32([0.05]), "zero_points": np.int32([0]), "host_scales": np.float32([0.05]),
            "host_zero_points": np.int32([0]), "quantization_dimension": None, "storage_min": -128, "storage_max": 127}
    y = torch.empty(n * n, dtype=torch.int8, device="cuda")
    hf.quant_fusion(x, [n, n], qin, [0, 1], y, out_dtype="s8", out_q=qout)
    torch.cuda.synchronize()
    rs = np.random.default_rng(82)
    i = np.concatenate([rs.integers(0, n, 3072), np.full(1024, n - 1)])
    j = np.concatenate([rs.integers(0, n, 3072), rs.integers(0, n, 1024)])
    codes = x[torch.from_numpy(i * n + j).cuda()].cpu().numpy()
    got = y[torch.from_numpy(j * n + i).cuda()].cpu().numpy()  # output element [i, j] sits at j*n + i
    in_spec = {"scales": scales, "zero_points": zps, "quantization_dimension": 1, "storage_min": -128,
               "storage_max": 127}
    out_spec = {"scales": np.float32([0.05]), "zero_points": np.int32([0]), "quantization_dimension": None,
                "storage_min": -128, "storage_max": 127}
    ref = np.array([oracle.quantize(out_spec, oracle.dequantize(in_spec, int(c), [int(a), int(b)]))
                    for c, a, b in zip(codes, i, j)])
    assert np.array_equal(got.astype(np.int64), ref.astype(np.int64))
    del x, y
    torch.cuda.empty_cache()


def test_bcast_exp_row_reduce_beyond_2_to_31_elements():
    """add(exp(x), broadcast(b)) reduced along rows of bf16[131080, 16384] (2.15e9 elements, the
    streaming row kernel): 32 sampled rows, the last ones among them, against the oracle within the
    reduction tolerance."""
    rows, cols = 131080, 16384
    g = inp.rng(83)
    x = _fill_device(rows * cols, lambda m: inp.normal_bf16(g, m).view(np.int16), torch.int16)
    b = inp.uniform_bf16(g, cols, -1.0, 1.0)
    bd = torch.from_numpy(b.view(np.int16)).cuda()
    out = torch.empty(rows, dtype=torch.float32, device="cuda")
    pro = {"ops": ["exp", "add_bcast"], "round_each": True,
           "bcast": {"tensor": bd, "dims": [cols], "dtype": "bf16", "broadcast_dimensions": [1]}}
    hf.reduce_fusion(x, [rows, cols], "bf16", [1], "add", 0.0, out, "f32", prologue=pro)
    torch.cuda.synchronize()
    rs = np.concatenate([np.random.default_rng(84).integers(0, rows, 28), np.arange(rows - 4, rows)])
    sub = x.view(rows, cols)[torch.from_numpy(rs).cuda()].contiguous().cpu().numpy().view(np.uint16)
    opro = {"ops": ["exp", "add_bcast"], "round_each": True,
            "bcast": {"data": b, "dims": [cols], "m2m": [0], "dtype": "bf16", "broadcast_dimensions": [1]}}
    ref, asum = oracle.reduce(sub.reshape(-1), [len(rs), cols], "bf16", [1], "add", 0.0, "f32", prologue=opro,
                              want_abs_sum=True)
    got = out.cpu().numpy()[rs].astype(np.float64)
    assert np.all(np.abs(got - ref.astype(np.float64)) <= 1e-5 * asum + 1e-6)
    del x
    torch.cuda.empty_cache()


# ---- more shapes through the same kernels -----------------------------------------------------------
@pytest.mark.parametrize("rows,cols", [(1, 1), (1, 7), (5, 3), (3, 4096 + 8), (2, 100003), (1000, 24)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_row_reduce_shapes(rows, cols, dtype):
    g = inp.rng(rows * 7 + cols)
    n = rows * cols
    data = inp.uniform_f32(g, n, -1, 1) if dtype == "f32" else inp.normal_bf16(g, n)
    for kind, init in (("add", 0.0), ("max", -math.inf), ("add", 2.5)):
        f = inp.Fusion(name="row", kind="reduce", dims=[rows, cols], m2m=[1, 0], dtype=dtype, data=data,
                       dimensions=[1], reduce_kind=kind, init=init,
                       prologue={"ops": ["exp"], "round_each": True} if kind == "add" else None,
                       out_dims=[rows], out_m2m=[0], out_dtype="f32")
        ref, asum = run_oracle(f)
        check(f, run_gpu(f), ref, asum)


@pytest.mark.parametrize("rows,cols,dtype", [(1, 1 << 22, "f32"), (3, 1000003, "f32"), (10, 1 << 20, "bf16"),
                                             (1, 65536 * 3 + 5, "bf16"), (150, 40000, "f32")])
def test_split_row_reduce(rows, cols, dtype):
    """Few long rows: the rows are cut into segments reduced by separate blocks into the workspace,
    then combined per row in segment order (with and without a prologue, add and max); the same results
    without a workspace (unsplit)."""
    g = inp.rng(rows + cols)
    n = rows * cols
    data = inp.uniform_f32(g, n, -1, 1) if dtype == "f32" else inp.normal_bf16(g, n)
    assert hf.reduce_workspace_size([rows, cols], dtype, [1]) > 0
    for kind, init, ops in (("add", 0.0, ["exp"]), ("max", -math.inf, None), ("add", 2.5, None),
                            ("max", -math.inf, ["neg", "exp"])):
        f = inp.Fusion(name="split", kind="reduce", dims=[rows, cols], m2m=[1, 0], dtype=dtype, data=data,
                       dimensions=[1], reduce_kind=kind, init=init,
                       prologue={"ops": ops, "round_each": True} if ops else None,
                       out_dims=[rows], out_m2m=[0], out_dtype="f32")
        ref, asum = run_oracle(f)
        d = DeviceFusion(f)
        assert d.workspace is not None
        d.run()
        torch.cuda.synchronize()
        check(f, d.output_numpy(), ref, asum)
        d.workspace = None  # unsplit
        d.run()
        torch.cuda.synchronize()
        check(f, d.output_numpy(), ref, asum)


def test_split_row_reduce_with_broadcast_and_layout():
    """A split reduce of add(exp(x), broadcast(b)) over the minor dims of a {0,1,2} layout array."""
    g = inp.rng(71)
    d0, d1 = 2, 300001
    x = inp.normal_bf16(g, d0 * d1)
    b = inp.uniform_bf16(g, d1, -1, 1)
    f = inp.Fusion(name="splitb", kind="reduce", dims=[d1, 1, d0], m2m=[0, 1, 2], dtype="bf16", data=x,
                   dimensions=[0, 1], reduce_kind="add", init=0.0,
                   prologue={"ops": ["exp", "add_bcast"], "round_each": True,
                             "bcast": {"data": b, "dims": [d1], "m2m": [0], "dtype": "bf16",
                                       "broadcast_dimensions": [0]}},
                   out_dims=[d0], out_m2m=[0], out_dtype="f32")
    ref, asum = run_oracle(f)
    check(f, run_gpu(f), ref, asum)


@pytest.mark.parametrize("a,r,b", [(1, 1, 1), (1, 9, 5), (3, 33, 264), (2, 1000, 7), (1, 4097, 2048)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_col_reduce_shapes(a, r, b, dtype):
    g = inp.rng(a * 1000 + r + b)
    n = a * r * b
    data = inp.uniform_f32(g, n, -4, 4) if dtype == "f32" else inp.normal_bf16(g, n)
    for kind, init in (("max", -math.inf), ("add", 0.0)):
        f = inp.Fusion(name="col", kind="reduce", dims=[a, r, b], m2m=[2, 1, 0], dtype=dtype, data=data,
                       dimensions=[1], reduce_kind=kind, init=init, out_dims=[a, b], out_m2m=[1, 0],
                       out_dtype=dtype if kind == "max" else "f32")
        ref, asum = run_oracle(f)
        check(f, run_gpu(f), ref, asum)


def test_reduce_general_patterns_and_layouts():
    g = inp.rng(99)
    dims = [4, 6, 5, 3]
    data = inp.uniform_f32(g, int(np.prod(dims)), -2, 2)
    cases = [([0, 2], [3, 2, 1, 0], [1, 0]), ([1, 3], [0, 1, 2, 3], [0, 1]), ([0, 1, 2, 3], [2, 0, 3, 1], []),
             ([2], [1, 3, 0, 2], [0, 2, 1]), ([3, 0], [3, 2, 1, 0], [1, 0]), ([], [3, 2, 1, 0], [3, 2, 1, 0])]
    for dimsred, m2m, out_m2m in cases:
        kept = [d for d in range(4) if d not in dimsred]
        for kind, init in (("add", 0.0), ("max", -math.inf)):
            f = inp.Fusion(name="gen", kind="reduce", dims=dims, m2m=m2m, dtype="f32", data=data,
                           dimensions=dimsred, reduce_kind=kind, init=init,
                           prologue={"ops": ["abs", "log"]} if kind == "add" else None,
                           out_dims=[dims[d] for d in kept], out_m2m=out_m2m, out_dtype="f32")
            ref, asum = run_oracle(f)
            check(f, run_gpu(f), ref, asum)


def test_reduce_empty_and_unit():
    z = np.zeros(0, np.float32)
    f = inp.Fusion(name="e", kind="reduce", dims=[4, 0], m2m=[1, 0], dtype="f32", data=z, dimensions=[1],
                   reduce_kind="add", init=1.5, out_dims=[4], out_m2m=[0], out_dtype="f32")
    ref, asum = run_oracle(f)
    check(f, run_gpu(f), ref, asum)
    f = inp.Fusion(name="e", kind="reduce", dims=[0, 5], m2m=[1, 0], dtype="f32", data=z, dimensions=[1],
                   reduce_kind="add", init=1.5, out_dims=[0], out_m2m=[0], out_dtype="f32")
    assert run_gpu(f).size == 0


def test_max_nan_and_signed_zero():
    rows, cols = 8, 64
    x = np.zeros((rows, cols), np.float32)
    x[0, 5] = np.nan
    x[1] = -0.0
    x[1, 7] = 0.0
    x[2] = -0.0
    x[3, :] = -np.inf
    x[4, 9] = np.inf
    for dims, red, data in (([rows, cols], [1], x.ravel()), ([cols, rows], [0], x.T.copy().ravel())):
        f = inp.Fusion(name="m", kind="reduce", dims=dims, m2m=[1, 0], dtype="f32", data=data, dimensions=red,
                       reduce_kind="max", init=-math.inf, out_dims=[rows], out_m2m=[0], out_dtype="f32")
        ref, _ = run_oracle(f)
        gpu = run_gpu(f)
        check(f, gpu, ref, None)
        assert np.isnan(gpu[0]) and gpu[1] == 0 and not np.signbit(gpu[1]) and np.signbit(gpu[2])


@pytest.mark.parametrize("d3", [8192 + 8, 20000, 16384])
def test_streaming_row_reduce_chunking(d3):
    """Rows long enough for the bulk-copy ring: a second chunk of 16 bytes, three chunks (broadcast read
    from memory), and exactly two full chunks (broadcast held in registers)."""
    f = inp.bcast_exp_reduce(seed=9, d0=2, d2=37, d3=d3)
    ref, asum = run_oracle(f)
    check(f, run_gpu(f), ref, asum)
    g = inp.rng(d3)
    x = inp.normal_bf16(g, 70 * d3)
    f = inp.Fusion(name="maxrow", kind="reduce", dims=[70, d3], m2m=[1, 0], dtype="bf16", data=x, dimensions=[1],
                   reduce_kind="max", init=-math.inf, out_dims=[70], out_m2m=[0], out_dtype="bf16")
    ref, asum = run_oracle(f)
    check(f, run_gpu(f), ref, asum)


def _reduce_case(name, data, dims, dtype, dimensions, kind, ops, init=0.0, round_each=True, out_dtype="f32"):
    kept = [d for d in range(len(dims)) if d not in dimensions]
    out_dims = [dims[d] for d in kept]
    return inp.Fusion(name=name, kind="reduce", dims=dims, m2m=list(range(len(dims) - 1, -1, -1)), dtype=dtype,
                      data=data, dimensions=dimensions, reduce_kind=kind, init=init,
                      prologue={"ops": ops, "round_each": round_each} if ops else None,
                      out_dims=out_dims, out_m2m=list(range(len(out_dims) - 1, -1, -1)), out_dtype=out_dtype)


# row (short rows), row (bulk-copy stream), column, general
REDUCE_PATTERNS = [([64, 1000], [1]), ([64, 8192], [1]), ([300, 64], [0]), ([4, 5, 6], [0, 2])]


@pytest.mark.parametrize("dims,dimensions", REDUCE_PATTERNS)
@pytest.mark.parametrize("dtype,round_each", [("f32", True), ("bf16", True), ("bf16", False)])
def test_max_of_exp_chains_bit_exact(dims, dimensions, dtype, round_each):
    """A max body keeps every term exact, so exp in the prologue is correctly rounded there (to the
    element type, or to f32 for f32 intermediates) and the result is bit-exact."""
    g = inp.rng(31)
    n = int(np.prod(dims))
    x = g.uniform(-20, 20, n).astype(np.float32)
    data = x if dtype == "f32" else inp.f32_to_bf16_bits(x)
    for ops in (["exp"], ["neg", "exp"]):
        f = _reduce_case("maxexp", data, dims, dtype, dimensions, "max", ops, init=-math.inf, round_each=round_each)
        ref, asum = run_oracle(f)
        check(f, run_gpu(f), ref, asum)


@pytest.mark.parametrize("dims,dimensions", REDUCE_PATTERNS)
def test_exp_inside_longer_chains_of_add_reductions(dims, dimensions):
    """exp followed by more ops is correctly rounded: exp -> log keeps tiny results (x down to -100, where
    exp is subnormal), and exp -> add_const(-1) near 0 cancels to about x, both within the tolerance."""
    g = inp.rng(37)
    n = int(np.prod(dims))
    deep = g.uniform(-100, -88, n).astype(np.float32)
    f = _reduce_case("explog", deep, dims, "f32", dimensions, "add", ["exp", "log"])
    ref, asum = run_oracle(f)
    check(f, run_gpu(f), ref, asum)
    near0 = g.uniform(-1e-3, 1e-3, n).astype(np.float32)
    f = _reduce_case("expm1", near0, dims, "f32", dimensions, "add", ["exp", ("add_const", -1.0)])
    ref, asum = run_oracle(f)
    check(f, run_gpu(f), ref, asum)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_reduce_init_rounded_to_the_input_type(dtype):
    """reduce (C2): init 0.1 is a value of the input element type."""
    g = inp.rng(3)
    x = g.uniform(-1, 1, 40 * 33).astype(np.float32)
    data = {"f32": x, "bf16": inp.f32_to_bf16_bits(x), "f16": x.astype(np.float16).view(np.uint16)}[dtype]
    for dims, dimensions in [([40, 33], [1]), ([40, 33], [0]), ([40, 0], [1])]:
        d = data[: int(np.prod(dims))]
        for kind in ("add", "max"):
            f = _reduce_case("init01", d, dims, dtype, dimensions, kind, None, init=0.1)
            ref, asum = run_oracle(f)
            check(f, run_gpu(f), ref, asum)


def test_bcast_row_reduce_variants():
    g = inp.rng(5)
    d0, d2, d3 = 2, 7, 515
    x = inp.normal_bf16(g, d0 * d2 * d3)
    b = inp.uniform_bf16(g, d3, -1, 1)
    for round_each in (True, False):
        f = inp.bcast_exp_reduce(seed=5, d0=d0, d2=d2, d3=d3)
        f.prologue = dict(f.prologue)
        f.prologue["round_each"] = round_each
        ref, asum = run_oracle(f)
        check(f, run_gpu(f), ref, asum)
    # broadcast along a kept dimension (one value per row)
    bk = inp.uniform_bf16(g, d2, -1, 1)
    f = inp.Fusion(name="perrow", kind="reduce", dims=[d0, 1, d2, d3], m2m=[3, 2, 0, 1], dtype="bf16", data=x,
                   dimensions=[3], reduce_kind="add", init=0.0,
                   prologue={"ops": ["add_bcast", "exp"], "round_each": True,
                             "bcast": {"data": bk, "dims": [d2], "m2m": [0], "dtype": "bf16",
                                       "broadcast_dimensions": [2]}},
                   out_dims=[d0, 1, d2], out_m2m=[2, 1, 0], out_dtype="f32")
    ref, asum = run_oracle(f)
    check(f, run_gpu(f), ref, asum)
    del b


# ---- transposes -----------------------------------------------------------------------------------------
@pytest.mark.parametrize("n", [1, 2, 4, 63, 64, 65, 68, 130, 132, 257, 1028])
def test_selfadd_log_sizes(n):
    f = inp.transpose_log(seed=n, n=n)
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)


@pytest.mark.parametrize("n", [192, 196])
@pytest.mark.parametrize("value", [1.015741229057312, 1.0, 0.5, 2.0 ** -130])
def test_selfadd_every_element_open(value, n):
    """Inputs whose log the first pass cannot round: the per-block list overflows and the per-thread
    spill path settles the rest (and exactly 1.0 / a subnormal take the special-operand route)."""
    data = np.full(n * n, value, dtype=np.float32)
    data[::7] = np.float32(1.3)  # a mix of open and settled elements
    f = inp.Fusion(name="open", kind="transpose", dims=[n, n], m2m=[1, 0], dtype="f32", data=data,
                   permutation=[1, 0], self_add=True, prologue={"ops": ["log"]}, out_dims=[n, n], out_m2m=[1, 0],
                   out_dtype="f32")
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)
    # the same value through the identity-layout log kernel
    x = torch.full((1024,), value, dtype=torch.float32, device="cuda")
    y = torch.empty_like(x)
    hf.transpose_fusion(x, [1024], "f32", [0], y, prologue={"ops": ["log"]})
    torch.cuda.synchronize()
    assert np.all(y.cpu().numpy() == np.float32(oracle.log(float(np.float32(value)), "f32")))


@pytest.mark.parametrize("n", [70, 72])
def test_selfadd_other_forms(n):
    g = inp.rng(8)
    data = inp.uniform_f32(g, n * n, 0.1, 3.0)
    for m2m in ([1, 0], [0, 1]):
        for pro, epi in ((None, None), ({"ops": ["log", "neg"]}, {"ops": ["abs"]})):
            f = inp.Fusion(name="sa", kind="transpose", dims=[n, n], m2m=m2m, dtype="f32", data=data,
                           permutation=[1, 0], self_add=True, prologue=pro, epilogue=epi, out_dims=[n, n],
                           out_m2m=m2m, out_dtype="f32")
            ref, _ = run_oracle(f)
            check(f, run_gpu(f), ref, None)
    # self add with different layouts (general path) and rank 3 with unit dims
    f = inp.Fusion(name="sa2", kind="transpose", dims=[n, n], m2m=[1, 0], dtype="f32", data=data, permutation=[1, 0],
                   self_add=True, prologue={"ops": ["log"]}, out_dims=[n, n], out_m2m=[0, 1], out_dtype="f32")
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)
    f = inp.Fusion(name="sa3", kind="transpose", dims=[n, 1, n], m2m=[2, 1, 0], dtype="f32", data=data,
                   permutation=[2, 1, 0], self_add=True, prologue={"ops": ["log"]}, out_dims=[n, 1, n],
                   out_m2m=[2, 1, 0], out_dtype="f32")
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "s8", "s32"])
def test_transpose_rank3_all_perms_and_layouts(dtype):
    import itertools

    g = inp.rng(17)
    dims = [5, 40, 33]
    n = int(np.prod(dims))
    if dtype == "f32":
        data = inp.uniform_f32(g, n, -10, 10)
    elif dtype == "bf16":
        data = inp.normal_bf16(g, n)
    elif dtype == "s8":
        data = inp.integers(g, n, -128, 127, np.int8)
    else:
        data = inp.integers(g, n, -2 ** 31, 2 ** 31 - 1, np.int32)
    layouts = [list(p) for p in itertools.permutations(range(3))]
    for pi, perm in enumerate(itertools.permutations(range(3))):
        for m2m in (layouts[pi], layouts[(pi + 2) % 6]):
            out_m2m = layouts[(pi + 3) % 6]
            f = inp.Fusion(name="t3", kind="transpose", dims=dims, m2m=m2m, dtype=dtype, data=data,
                           permutation=list(perm), out_dims=[dims[p] for p in perm], out_m2m=out_m2m,
                           out_dtype=dtype)
            ref, _ = run_oracle(f)
            check(f, run_gpu(f), ref, None)


def test_transpose_emitter_example_exp_abs():
    """The transpose-emitter example: f32[20,160,170] -> exp -> transpose {2,1,0} -> abs, bit-exact (exp
    is correctly rounded on both sides)."""
    g = inp.rng(21)
    dims = [20, 160, 170]
    data = inp.uniform_f32(g, int(np.prod(dims)), -3, 3)
    f = inp.Fusion(name="emit", kind="transpose", dims=dims, m2m=[2, 1, 0], dtype="f32", data=data,
                   permutation=[2, 1, 0], prologue={"ops": ["exp"]}, epilogue={"ops": ["abs"]},
                   out_dims=[170, 160, 20], out_m2m=[2, 1, 0], out_dtype="f32")
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)


@pytest.mark.parametrize("dims,perm", [([36, 20, 68], [2, 1, 0]), ([132, 72], [1, 0]), ([4, 12, 8, 132], [3, 0, 2, 1]),
                                       ([8, 4, 12, 4, 68], [4, 2, 0, 3, 1]), ([200, 3, 76], [2, 0, 1])])
def test_transpose_tensor_copy_tiles(dims, perm):
    """Shapes whose strides allow the tensor-copy tile kernel (4-byte elements, strides multiples of four):
    ragged 64 x 64 tiles and one to three batch axes; f32 with prologue / epilogue chains and s32 without,
    bit-exact against the oracle."""
    g = inp.rng(sum(dims))
    n = int(np.prod(dims))
    out_dims = [dims[q] for q in perm]
    m2m, out_m2m = list(range(len(dims) - 1, -1, -1)), list(range(len(dims) - 1, -1, -1))
    x = inp.uniform_f32(g, n, -3, 3)
    for pro, epi in ((["exp"], ["abs"]), (None, None), (["neg", ("mul_const", 0.37), "tanh"], [("add_const", 1.5)])):
        f = inp.Fusion(name="tt", kind="transpose", dims=dims, m2m=m2m, dtype="f32", data=x, permutation=perm,
                       prologue={"ops": pro, "round_each": True} if pro else None,
                       epilogue={"ops": epi, "round_each": True} if epi else None,
                       out_dims=out_dims, out_m2m=out_m2m, out_dtype="f32")
        ref, asum = run_oracle(f)
        check(f, run_gpu(f), ref, asum)
    xi = g.integers(-2 ** 31, 2 ** 31 - 1, size=n, dtype=np.int64).astype(np.int32)
    f = inp.Fusion(name="tti", kind="transpose", dims=dims, m2m=m2m, dtype="s32", data=xi, permutation=perm,
                   out_dims=out_dims, out_m2m=out_m2m, out_dtype="s32")
    ref, asum = run_oracle(f)
    check(f, run_gpu(f), ref, asum)


def test_transpose3_exp_abs_full_size():
    """The transpose-emitter fusion scaled up (f32[512,640,680] -> [680,640,512]) as the benchmark runs
    it, on every output."""
    f = inp.transpose3_exp_abs(seed=1)
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)


def _gpu_exp_bits(first: int, count: int) -> np.ndarray:
    x = torch.arange(first, first + count, dtype=torch.int64, device="cuda").to(torch.int32).view(torch.float32)
    y = torch.empty_like(x)
    hf.transpose_fusion(x, [count], "f32", [0], y, prologue={"ops": ["exp"]})
    torch.cuda.synchronize()
    return y.view(torch.int32).cpu().numpy().view(np.uint32)


def test_exp_exhaustive():
    """Every f32 whose exp is neither 0 nor inf after rounding, both signs (x in [-104, 89]), plus the
    ends of the range, bit-exact against the oracle's correctly rounded exp."""
    chunk = 1 << 27
    total_bad, examples = 0, []
    for lo, hi in ((0x00000000, 0x42B20000), (0x80000000, 0xC2D00000)):  # +0 .. 89.0, -0 .. -104.0
        for first in range(lo, hi, chunk):
            n = min(chunk, hi - first)
            start = first - (1 << 32) if first >= 1 << 31 else first
            bad, ex = oracle.check_exp_f32(first, _gpu_exp_bits(start, n))
            total_bad += bad
            examples += ex
    for first in (0x42B20000, 0x7F7F0000, 0x7F800000, 0xC2D00000, 0xFF7F0000, 0xFF800000):  # past the range
        start = first - (1 << 32) if first >= 1 << 31 else first
        bad, ex = oracle.check_exp_f32(first, _gpu_exp_bits(start, 1 << 16))
        total_bad += bad
        examples += ex
    assert total_bad == 0, [hex(v) for v in examples[:16]]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "s8"])
def test_layout_convert_rank4(dtype):
    import itertools

    g = inp.rng(3)
    dims = [3, 1, 37, 66]
    n = int(np.prod(dims))
    data = (inp.uniform_f32(g, n, -1, 1) if dtype == "f32" else
            inp.normal_bf16(g, n) if dtype == "bf16" else inp.integers(g, n, -128, 127, np.int8))
    for m2m in ([3, 2, 1, 0], [0, 1, 2, 3], [3, 2, 0, 1]):
        for out_m2m in itertools.islice(itertools.permutations(range(4)), 0, 24, 5):
            f = inp.Fusion(name="lc", kind="layout", dims=dims, m2m=m2m, dtype=dtype, data=data, out_dims=dims,
                           out_m2m=list(out_m2m), out_dtype=dtype)
            ref, _ = run_oracle(f)
            check(f, run_gpu(f), ref, None)


def test_unaligned_pointers():
    """Operands that start 1 element past an aligned address take the narrow-access variants."""
    g = inp.rng(4)
    rows, cols = 33, 520
    base = torch.from_numpy(inp.uniform_f32(g, rows * cols + 1, -1, 1)).cuda()
    x = base[1:]
    out = torch.empty(rows + 1, dtype=torch.float32, device="cuda")[1:]
    hf.reduce_fusion(x, [rows, cols], "f32", [1], "add", 0.0, out, "f32", prologue={"ops": ["exp"]})
    f = inp.Fusion(name="u", kind="reduce", dims=[rows, cols], m2m=[1, 0], dtype="f32", data=x.cpu().numpy(),
                   dimensions=[1], reduce_kind="add", init=0.0, prologue={"ops": ["exp"]}, out_dims=[rows],
                   out_m2m=[0], out_dtype="f32")
    ref, asum = run_oracle(f)
    torch.cuda.synchronize()
    check(f, out.cpu().numpy(), ref, asum)
    n = 68
    p = torch.from_numpy(inp.uniform_f32(g, n * n + 1, 0.5, 2)).cuda()[1:]
    o = torch.empty(n * n + 1, dtype=torch.float32, device="cuda")[1:]
    hf.transpose_fusion(p, [n, n], "f32", [1, 0], o, prologue={"ops": ["log"]}, self_add=True)
    f = inp.Fusion(name="u2", kind="transpose", dims=[n, n], m2m=[1, 0], dtype="f32", data=p.cpu().numpy(),
                   permutation=[1, 0], self_add=True, prologue={"ops": ["log"]}, out_dims=[n, n], out_m2m=[1, 0],
                   out_dtype="f32")
    ref, _ = run_oracle(f)
    torch.cuda.synchronize()
    check(f, o.cpu().numpy(), ref, None)


# ---- quantized relayout ----------------------------------------------------------------------------------
def _qspec(g, n, per_axis_dim, smin=-128, smax=127):
    if per_axis_dim is None:
        return {"scales": np.array([np.float32(g.uniform(0.01, 0.2))], np.float32),
                "zero_points": np.array([int(g.integers(-5, 6))], np.int32), "quantization_dimension": None,
                "storage_min": smin, "storage_max": smax}
    return {"scales": inp.uniform_f32(g, n, 0.001, 0.1), "zero_points": inp.integers(g, n, -20, 20, np.int32),
            "quantization_dimension": per_axis_dim, "storage_min": smin, "storage_max": smax}


@pytest.mark.parametrize("n0,n1", [(128, 128), (256, 384), (384, 128), (130, 200), (7, 3), (4096, 16)])
def test_quant_relayout_variants(n0, n1):
    g = inp.rng(n0 + n1)
    q = inp.integers(g, n0 * n1, -128, 127, np.int8)
    dims = [n0, n1]
    for qin_dim, qout_dim in ((1, None), (0, None), (None, None), (1, 0), (None, 1)):
        qin = _qspec(g, dims[qin_dim] if qin_dim is not None else 1, qin_dim)
        qout = _qspec(g, dims[qout_dim] if qout_dim is not None else 1, qout_dim, smin=-100, smax=90)
        for out_m2m in ([0, 1], [1, 0]):
            f = inp.Fusion(name="q", kind="quant", dims=dims, m2m=[1, 0], dtype="s8", data=q, in_q=qin,
                           out_q=qout, out_dims=dims, out_m2m=out_m2m, out_dtype="s8")
            ref, _ = run_oracle(f)
            check(f, run_gpu(f), ref, None)
    # float output and a float op between dequantize and quantize
    qin = _qspec(g, n1, 1)
    f = inp.Fusion(name="qf", kind="quant", dims=dims, m2m=[1, 0], dtype="s8", data=q, in_q=qin, out_q=None,
                   out_dims=dims, out_m2m=[0, 1], out_dtype="f32")
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)
    f = inp.Fusion(name="qn", kind="quant", dims=dims, m2m=[1, 0], dtype="s8", data=q, in_q=qin,
                   out_q=_qspec(g, 1, None), prologue={"ops": ["neg", "abs"]}, out_dims=dims, out_m2m=[0, 1],
                   out_dtype="s8")
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)


def test_quant_division_ties():
    """Reals that land exactly on half-integers after division take the exact-division branch and round
    to even: scale_in = scale_out * k/2 for odd k."""
    n0, n1 = 256, 256
    g = inp.rng(6)
    q = inp.integers(g, n0 * n1, -128, 127, np.int8)
    qin = {"scales": np.full(n1, 0.025, np.float32), "zero_points": np.zeros(n1, np.int32),
           "quantization_dimension": 1}
    qout = {"scales": np.array([0.05], np.float32), "zero_points": np.array([0], np.int32),
            "quantization_dimension": None}
    f = inp.Fusion(name="qt", kind="quant", dims=[n0, n1], m2m=[1, 0], dtype="s8", data=q, in_q=qin, out_q=qout,
                   out_dims=[n0, n1], out_m2m=[0, 1], out_dtype="s8")
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)


@pytest.mark.parametrize("ratio", [3000.0, 20000.0])
def test_quant_scale_ratios(ratio):
    """Input/output scale ratios that push quotients far past the i8 range, so that saturation decides
    (3000), and beyond the range the bracketed fast test accepts (20000: the exact test decides)."""
    n0, n1 = 256, 384
    g = inp.rng(int(ratio))
    q = inp.integers(g, n0 * n1, -128, 127, np.int8)
    for qin_dim, qout_dim, smin, smax in ((1, None, -128, 127), (0, 1, -128, 127), (None, None, -7, 9)):
        dims = [n0, n1]
        nin = dims[qin_dim] if qin_dim is not None else 1
        nout = dims[qout_dim] if qout_dim is not None else 1
        scale_out = inp.uniform_f32(g, nout, 0.5, 1.0) / np.float32(ratio)
        qin = {"scales": inp.uniform_f32(g, nin, 0.5, 1.0), "zero_points": inp.integers(g, nin, -20, 20, np.int32),
               "quantization_dimension": qin_dim}
        qout = {"scales": scale_out.astype(np.float32), "zero_points": inp.integers(g, nout, -3, 3, np.int32),
                "quantization_dimension": qout_dim, "storage_min": smin, "storage_max": smax}
        f = inp.Fusion(name="qr", kind="quant", dims=dims, m2m=[1, 0], dtype="s8", data=q, in_q=qin, out_q=qout,
                       out_dims=dims, out_m2m=[0, 1], out_dtype="s8")
        ref, _ = run_oracle(f)
        out = run_gpu(f)
        check(f, out, ref, None)
        assert np.count_nonzero(ref == smax) > 0 and np.count_nonzero(ref == smin) > 0


# ---- the correctly rounded log ------------------------------------------------------------------------------
def _gpu_log_bits(first: int, count: int) -> np.ndarray:
    x = torch.arange(first, first + count, dtype=torch.int64, device="cuda").to(torch.int32).view(torch.float32)
    y = torch.empty_like(x)
    hf.transpose_fusion(x, [count], "f32", [0], y, prologue={"ops": ["log"]})
    torch.cuda.synchronize()
    return y.view(torch.int32).cpu().numpy().view(np.uint32)


def test_log_exhaustive_on_the_input_range():
    """Every f32 in [0.5, 2) -- the range the transpose workload draws from -- bit-exact."""
    first, last = 0x3F000000, 0x40000000
    bad, examples = oracle.check_log_f32(first, _gpu_log_bits(first, last - first))
    assert bad == 0, [hex(v) for v in examples]


def test_log_exhaustive_all_floats():
    """Every f32 bit pattern with the sign bit clear (zero, subnormals, normals, inf, NaNs), bit-exact;
    and a sample of negative inputs (NaN)."""
    chunk = 1 << 27
    total_bad = 0
    examples = []
    for first in range(0, 1 << 31, chunk):
        bad, ex = oracle.check_log_f32(first, _gpu_log_bits(first, chunk))
        total_bad += bad
        examples += ex
    assert total_bad == 0, [hex(v) for v in examples[:16]]
    bad, ex = oracle.check_log_f32(0x80000000, _gpu_log_bits(0x80000000 - (1 << 32), 1 << 20))
    assert bad == 0


# ---- loop fusions: chains with tanh, constants and the input as operands (XLA:GPU Emitters, "Loop
# emitter"); 16-bit results correctly rounded, so bit-exact -------------------------------------------------
def _chain_fusion(data, dtype, ops, name="chain"):
    n = len(data)
    return inp.Fusion(name=name, kind="transpose", dims=[n], m2m=[0], dtype=dtype, data=data, permutation=[0],
                      prologue={"ops": ops, "round_each": True}, out_dims=[n], out_m2m=[0], out_dtype=dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("op", ["tanh", "exp", "log"])
def test_16bit_exp_log_tanh_every_input(dtype, op):
    """All 65536 bit patterns through the packed 16-bit kernel, then through the scalar kernel (an
    unaligned view), both against the oracle's correctly rounded values."""
    data = np.arange(1 << 16, dtype=np.uint16)
    f = _chain_fusion(data, dtype, [op])
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)
    base = torch.from_numpy(np.concatenate([[0], data]).astype(np.uint16).view(np.int16)).cuda()
    x = base[1:]
    y = torch.empty(len(data) + 1, dtype=torch.int16, device="cuda")[1:]
    hf.transpose_fusion(x, [len(data)], dtype, [0], y, prologue={"ops": [op], "round_each": True})
    torch.cuda.synchronize()
    check(f, y.cpu().numpy().view(np.uint16), ref, None)


def test_gelu_every_bf16_input():
    data = np.arange(1 << 16, dtype=np.uint16)
    f = inp.gelu_bf16(dims=[1 << 16], data=data)
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)


@pytest.mark.parametrize("dims", [[6, 512, 4096], [3, 7, 1001]])
def test_gelu_loop_fusion_sizes(dims):
    """The emitter's GELU at its size (the benchmark's launch), and a ragged one (tail elements)."""
    f = inp.gelu_bf16(seed=3, dims=dims)
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)


@pytest.mark.parametrize("dtype,ops", [("bf16", list(inp.GELU_CHAIN)),
                                       ("f16", ["exp", ("mul_const", 0.5), "tanh", "log"])])
def test_chain_table_every_16bit_input(dtype, ops):
    """Inputs large enough for the table kernel (16-bit chains of 2^22 elements or more): every bit
    pattern 64 times over plus a ragged tail, bit-exact against the oracle."""
    pats = np.arange(1 << 16, dtype=np.uint16)
    data = np.concatenate([np.tile(pats, 64), pats[:13]])
    f = _chain_fusion(data, dtype, ops)
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)
    # f32 intermediates (one rounding at the end): the table is built with the per-element code
    n = len(data)
    f = inp.Fusion(name="chain_f32mid", kind="transpose", dims=[n], m2m=[0], dtype=dtype, data=data, permutation=[0],
                   prologue={"ops": ops, "round_each": False}, out_dims=[n], out_m2m=[0], out_dtype=dtype)
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)


@pytest.mark.parametrize("dtype,ops", [
    ("bf16", list(inp.GELU_CHAIN)),  # one run table: multiply, tanh, add 1, multiply
    ("bf16", ["neg", ("add_const", 0.75), "tanh", "abs", ("mul_const", -3.0), "mul_input"]),  # run table
    ("bf16", ["mul_input", "tanh", "add_input", "tanh", ("mul_const", 2.0), "mul_input"]),  # two tanh runs: tanh table
    ("bf16", ["mul_input", "tanh", "add_input"]),  # a lone tanh: tanh table
    ("f16", ["mul_input", ("add_const", -1.5), "neg", ("mul_const", 0.3), "add_input", "abs"]),  # no table
])
def test_generated_chain_kernels_every_16bit_input(dtype, ops):
    """Chains of 2^20 elements or more that the run-time generator covers (hlo_jit_kernels counts the
    kernels it built; -1 would mean NVRTC is unavailable on the GPU machine): every bit pattern 64 times over
    plus a ragged tail and an odd element count, bit-exact against the oracle."""
    pats = np.arange(1 << 16, dtype=np.uint16)
    for tail in (13, 8):
        data = np.concatenate([np.tile(pats, 64), pats[:tail]])
        f = _chain_fusion(data, dtype, ops)
        ref, _ = run_oracle(f)
        check(f, run_gpu(f), ref, None)
    assert hf.jit_kernels() >= 1


@pytest.mark.parametrize("dtype,ops", [
    ("bf16", list(inp.GELU_CHAIN)),
    ("f16", ["mul_input", ("add_const", -1.5), "neg", ("mul_const", 0.3), "add_input", "abs"]),
])
def test_generated_chain_kernels_many_chunks_per_block(dtype, ops):
    """2^26 + 5 elements: each block of the generated kernel streams far more 16 KiB chunks than its ring
    holds, so every stage is refilled many times (with and without the tanh table in shared memory), and
    five elements sit past the last whole vector. The chain is elementwise, so the oracle's value of each
    of the 65536 bit patterns, indexed by the input, is the expected output; bit-exact."""
    pats = np.arange(1 << 16, dtype=np.uint16)
    data = np.concatenate([np.tile(pats[np.random.default_rng(5).permutation(1 << 16)], 1 << 10), pats[:5]])
    per_pattern, _ = run_oracle(_chain_fusion(pats, dtype, ops))
    f = _chain_fusion(data, dtype, ops)
    check(f, run_gpu(f), np.asarray(per_pattern).reshape(-1)[data], None)
    assert hf.jit_kernels() >= 1


def test_generated_run_tables_past_the_last_slot_and_across_streams():
    """Twelve distinct bf16 chains whose tanh run becomes a 65536-entry table built on the device: more
    chains than the library keeps table slots for, so the later ones read the tanh table instead. Each
    chain's first launch goes to a side stream (the table is built there) and the second to the current
    stream (which must wait for that table). 2^20 + 3 elements, every bit pattern 16 times; bit-exact
    against the oracle's value of each pattern."""
    pats = np.arange(1 << 16, dtype=np.uint16)
    data = np.concatenate([np.tile(pats, 16), pats[:3]])
    side = torch.cuda.Stream()
    for k in range(12):
        ops = ["mul_input", ("mul_const", 0.25 + k / 16), "tanh", ("add_const", 1.0), "mul_input"]
        per_pattern, _ = run_oracle(_chain_fusion(pats, "bf16", ops))
        expected = np.asarray(per_pattern).reshape(-1)[data]
        f = _chain_fusion(data, "bf16", ops)
        d = DeviceFusion(f)
        torch.cuda.synchronize()  # the input's upload has landed
        with torch.cuda.stream(side):
            d.run(stream=side)
        side.synchronize()
        check(f, d.output_numpy(), expected, None)
        d.out.zero_()
        d.run()
        torch.cuda.synchronize()
        check(f, d.output_numpy(), expected, None)
    assert hf.jit_kernels() >= 12


@pytest.mark.parametrize("dtype,ops", [
    ("bf16", ["mul_input", ("mul_const", 0.3125), "tanh", ("add_const", 1.0), "mul_input"]),  # run table
    ("f16", ["mul_input", ("add_const", -2.5), "abs", "mul_input"]),  # no table
])
def test_generated_chains_under_graph_capture(dtype, ops):
    """A chain of 2^20 + 3 elements captured into a CUDA graph (torch.cuda.graph) on its first use, then
    captured again after it has run outside a capture: every replay gives the oracle's values (the
    first capture, and a chain with a run table, take the interpreter; the rest the generated kernel)."""
    pats = np.arange(1 << 16, dtype=np.uint16)
    data = np.concatenate([np.tile(pats, 16), pats[:3]])
    per_pattern, _ = run_oracle(_chain_fusion(pats, dtype, ops))
    expected = np.asarray(per_pattern).reshape(-1)[data]
    # the interpreter's one-time setup (table address, attributes) outside a capture
    warm = DeviceFusion(_chain_fusion(np.tile(pats, 4), dtype, ["tanh"] if dtype == "bf16" else ["abs"]))
    warm.run()
    f = _chain_fusion(data, dtype, ops)
    d = DeviceFusion(f)
    torch.cuda.synchronize()
    for plain_run_first in (False, True):
        if plain_run_first:
            d.run()
            torch.cuda.synchronize()
        d.out.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            d.run()
        d.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        check(f, d.output_numpy(), expected, None)


def test_gelu_chain_f32_bit_exact():
    """The same GELU chain on f32 (every op, tanh included, correctly rounded on both sides): bit-exact."""
    g = np.random.default_rng(13)
    x = np.concatenate([g.standard_normal(1 << 20), g.uniform(-12, 12, 1 << 16)]).astype(np.float32)
    f = _chain_fusion(x, "f32", list(inp.GELU_CHAIN))
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)


def _gpu_unary_bits(op: str, first: int, count: int) -> np.ndarray:
    x = torch.arange(first, first + count, dtype=torch.int64, device="cuda").to(torch.int32).view(torch.float32)
    y = torch.empty_like(x)
    hf.transpose_fusion(x, [count], "f32", [0], y, prologue={"ops": [op]})
    torch.cuda.synchronize()
    return y.view(torch.int32).cpu().numpy().view(np.uint32)


def test_f32_tanh_exhaustive():
    """Every f32 in [0, 10] (tanh rounds to 1 beyond 9.02; the GPU evaluates |x| and restores the sign),
    a run of negative inputs, and the ends of the range, bit-exact against the oracle's correctly
    rounded tanh."""
    chunk = 1 << 27
    total_bad, examples = 0, []
    hi = 0x41200000  # 10.0
    for first in range(0, hi, chunk):
        bad, ex = oracle.check_tanh_f32(first, _gpu_unary_bits("tanh", first, min(chunk, hi - first)))
        total_bad += bad
        examples += ex
    for first in (0xBF000000, 0x80000000, 0x7F7F0000, 0x7F800000, 0xFF7F0000, 0xFF800000):
        start = first - (1 << 32) if first >= 1 << 31 else first
        bad, ex = oracle.check_tanh_f32(first, _gpu_unary_bits("tanh", start, 1 << 20))
        total_bad += bad
        examples += ex
    assert total_bad == 0, [hex(v) for v in examples[:16]]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_longest_chain_of_exact_ops(dtype):
    """Sixteen ops (the most a chain holds) of IEEE add/multiply/negate/abs: bit-exact."""
    g = np.random.default_rng(12)
    x = g.standard_normal(50001).astype(np.float32)
    data = x if dtype == "f32" else inp.f32_to_bf16_bits(x)
    ops = ["mul_input", ("add_const", 0.25), ("mul_const", -1.5), "add_input", "abs", ("mul_const", 0.1),
           "mul_input", "neg", ("add_const", 3.0), "mul_input", ("mul_const", 0.7), "add_input", "abs",
           ("add_const", -2.0), "mul_input", "neg"]
    f = _chain_fusion(data, dtype, ops)
    ref, _ = run_oracle(f)
    check(f, run_gpu(f), ref, None)


# ---- variadic reduce with the max/argmax body (XLA Operation Semantics, "Variadic Reduce") ----------------
def _torch_buf(np_arr):
    a = np.ascontiguousarray(np_arr)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def _argmax_case(data, dims, dtype, dimensions, m2m=None, indices=None, idx_m2m=None, out_m2m=None, out_idx_m2m=None,
                 init_value=-math.inf, init_index=-1):
    ref_v, ref_i = oracle.reduce_max_argmax(data, dims, dtype, dimensions, init_value, init_index, m2m=m2m,
                                            out_m2m=out_m2m, indices=indices, idx_m2m=idx_m2m, out_idx_m2m=out_idx_m2m)
    n_out = ref_v.size
    x = _torch_buf(data)
    k = _torch_buf(indices) if indices is not None else None
    tdt = torch.float32 if dtype == "f32" else torch.int16
    ov = torch.empty(max(1, n_out), dtype=tdt, device="cuda")
    oi = torch.empty(max(1, n_out), dtype=torch.int32, device="cuda")
    hf.reduce_max_argmax(x, dims, dtype, dimensions, ov, oi, init_value=init_value, init_index=init_index, indices=k,
                         in_m2m=m2m, idx_m2m=idx_m2m, out_m2m=out_m2m, out_idx_m2m=out_idx_m2m)
    torch.cuda.synchronize()
    gv = ov.cpu().numpy()[:n_out]
    gi = oi.cpu().numpy()[:n_out]
    if dtype == "f32":
        same_v = (gv.view(np.uint32) == ref_v.view(np.uint32)) | (np.isnan(gv) & np.isnan(ref_v))
    else:
        same_v = gv.view(np.uint16) == np.asarray(ref_v, np.uint16)
    assert same_v.all(), f"{int((~same_v).sum())} values differ"
    assert np.array_equal(gi, ref_i), f"{int((gi != ref_i).sum())} indices differ, first at {np.flatnonzero(gi != ref_i)[:4]}"


def _values(g, n, dtype, ties=True):
    x = (g.integers(-4, 5, n) if ties else g.standard_normal(n)).astype(np.float32)
    x[g.integers(0, n, max(1, n // 97))] = np.nan
    x[g.integers(0, n, max(1, n // 89))] = -0.0
    if dtype == "bf16":
        return inp.f32_to_bf16_bits(x)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    return x


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("shape", [[37, 1000], [64, 1024], [5, 4096], [300, 7]])
def test_argmax_rows(dtype, shape):
    g = np.random.default_rng(shape[0] * 7 + shape[1])
    _argmax_case(_values(g, shape[0] * shape[1], dtype), shape, dtype, [1])
    _argmax_case(_values(g, shape[0] * shape[1], dtype, ties=False), shape, dtype, [1], init_value=0.5, init_index=-7)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_argmax_columns_layouts_and_given_indices(dtype):
    g = np.random.default_rng(31)
    dims = [6, 50, 33]
    n = int(np.prod(dims))
    data = _values(g, n, dtype)
    k = g.permutation(n).astype(np.int32)
    _argmax_case(data, [50, 33], dtype, [0], m2m=[1, 0])                       # reduce the major dim
    for dimsred, m2m, km2m, om2m in (([0, 2], [2, 1, 0], [0, 1, 2], [0]), ([1], [0, 2, 1], [2, 1, 0], [0, 1]),
                                     ([2, 0], [1, 0, 2], [1, 2, 0], [0]), ([0, 1, 2], [2, 1, 0], [2, 0, 1], [])):
        kept = [d for d in range(3) if d not in dimsred]
        _argmax_case(data, dims, dtype, dimsred, m2m=m2m, indices=k, idx_m2m=km2m, out_m2m=om2m,
                     out_idx_m2m=list(reversed(om2m)) if len(kept) == 2 else om2m)


def test_argmax_empty_and_degenerate():
    _argmax_case(np.zeros(0, np.float32), [4, 0], "f32", [1], init_index=-3)          # empty reduced dim
    _argmax_case(np.float32([np.nan] * 12), [3, 4], "f32", [1], init_value=1.0)        # all NaN: init stays
    _argmax_case(np.float32([2.0] * 12), [3, 4], "f32", [1], init_value=2.0, init_index=9)  # ties with init


def test_argmax_full_size_logits():
    """argmax over f32[4096, 32768] rows (the next-rows benchmark workload)."""
    f = inp.argmax_f32(seed=4)
    _argmax_case(f.data, f.dims, f.dtype, f.dimensions)


# ---- quantized elementwise binary ops (dequantize_op_quantize) ---------------------------------------------
def _qpt(scale, zp, smin=-128, smax=127):
    return {"scales": np.float32([scale]), "zero_points": np.int32([zp]), "quantization_dimension": None,
            "host_scales": np.float32([scale]), "host_zero_points": np.int32([zp]), "storage_min": smin,
            "storage_max": smax}


# Parameter sets: "packed" keeps every |r / s| small (the packed kernel for add, maximum, minimum and
# multiply; its clamp variant, then its saturating-pack one); "wide" scales push r / s past that kernel's
# range (the pair-table kernel for large inputs, the vector kernel for small ones).
QB_PARAMS = {
    "packed_clamp": (_qpt(0.0371, 4), _qpt(0.113, -9), _qpt(0.09, 2, -100, 120)),
    "packed": (_qpt(0.0371, 4), _qpt(0.113, -9), _qpt(0.0731, -3)),
    "wide": (_qpt(61.0, 4), _qpt(47.5, -9), _qpt(0.0013, 2, -100, 120)),
}


@pytest.mark.parametrize("params", list(QB_PARAMS))
@pytest.mark.parametrize("op", ["add", "divide", "maximum", "minimum", "multiply"])
def test_quant_binary_every_code_pair(op, params):
    """All 65536 code pairs, aligned (packed or vector kernel) and through unaligned views (per-element
    kernel)."""
    codes = np.arange(-128, 128, dtype=np.int8)
    a, b = np.repeat(codes, 256), np.tile(codes, 256)
    ql, qr, qo = QB_PARAMS[params]
    ref = oracle.quant_binary(op, a, b, [a.size], ql, qr, qo)
    for shift in (0, 1):
        base_a = torch.from_numpy(np.concatenate([np.zeros(shift, np.int8), a])).cuda()
        base_b = torch.from_numpy(np.concatenate([np.zeros(shift, np.int8), b])).cuda()
        out = torch.empty(a.size + shift, dtype=torch.int8, device="cuda")
        hf.quant_binary(op, base_a[shift:], base_b[shift:], [a.size], ql, qr, out[shift:], qo)
        torch.cuda.synchronize()
        got = out[shift:].cpu().numpy()
        assert np.array_equal(got, ref), f"{int((got != ref).sum())} codes differ (shift {shift})"


@pytest.mark.parametrize("params", list(QB_PARAMS))
@pytest.mark.parametrize("op", ["add", "divide", "maximum", "minimum", "multiply"])
def test_quant_binary_large_every_code_pair(op, params):
    """Inputs of 2^22 elements or more (the packed kernel, or the pair-table kernel for divide and for
    the wide parameters): all 65536 code pairs 64 times over plus a ragged tail, bit-exact against the
    oracle."""
    codes = np.arange(-128, 128, dtype=np.int8)
    a0, b0 = np.repeat(codes, 256), np.tile(codes, 256)
    a = np.concatenate([np.tile(a0, 64), a0[:13]])
    b = np.concatenate([np.tile(b0, 64), b0[7:20]])
    ql, qr, qo = QB_PARAMS[params]
    ref = oracle.quant_binary(op, a, b, [a.size], ql, qr, qo)
    out = torch.empty(a.size, dtype=torch.int8, device="cuda")
    hf.quant_binary(op, torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), [a.size], ql, qr, out, qo)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} codes differ"


def test_quant_binary_layouts_and_sizes():
    g = np.random.default_rng(41)
    dims = [37, 53, 5]
    n = int(np.prod(dims))
    a = g.integers(-128, 128, n).astype(np.int8)
    b = g.integers(-128, 128, n).astype(np.int8)
    q = _qpt(0.3, 0)
    for lm, rm, om in (([2, 1, 0], [0, 1, 2], [1, 2, 0]), ([0, 2, 1], [0, 2, 1], [0, 2, 1])):
        ref = oracle.quant_binary("add", a, b, dims, q, q, q, lhs_m2m=lm, rhs_m2m=rm, out_m2m=om)
        out = torch.empty(n, dtype=torch.int8, device="cuda")
        hf.quant_binary("add", torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), dims, q, q, out, q,
                        lhs_m2m=lm, rhs_m2m=rm, out_m2m=om)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), ref)


def test_quant_add_full_size():
    f = inp.quant_add_s8(seed=2)
    ref = oracle.quant_binary(f.op, f.data, f.rhs, f.dims, f.in_q, f.in_q, f.out_q)
    assert np.array_equal(run_gpu(f), ref)


# ---- device faults ---------------------------------------------------------------------------------------
def test_bounded_wait_reports_a_fault():
    """A bounded wait that runs out (one block waits about a millisecond on a barrier nothing completes)
    records HLO_FAULT_COPY_TIMEOUT; the context stays usable and the bit clears."""
    hf.device_faults(clear=True)
    assert hf.device_faults() == 0
    hf.selftest_bounded_wait()
    assert hf.device_faults(clear=True) == hf.FAULT_COPY_TIMEOUT
    assert hf.device_faults() == 0
    f = inp.small("row_reduce_exp", seed=1)  # the device still runs fusions afterwards
    ref, asum = run_oracle(f)
    check(f, run_gpu(f), ref, asum)
    assert hf.device_faults() == 0


# ---- quantized data movement: broadcast_in_dim and reshape -------------------------------------------------
def _to_physical(arr, m2m):
    return np.ascontiguousarray(np.transpose(arr, list(reversed(m2m)))).ravel()


def _qdev(q):
    """Device copies of per-axis parameters (host copies kept for the library's value checks)."""
    out = {"host_scales": np.float32(q["scales"]), "host_zero_points": np.int32(q["zero_points"]),
           "quantization_dimension": q.get("quantization_dimension")}
    if q.get("quantization_dimension") is not None:
        out["scales"] = torch.from_numpy(np.float32(q["scales"])).cuda()
        out["zero_points"] = torch.from_numpy(np.int32(q["zero_points"])).cuda()
    return out


def _gpu_quant_broadcast(codes_phys, dims, q, bdims, out_dims, in_m2m, out_m2m):
    x = torch.from_numpy(np.ascontiguousarray(codes_phys, np.int8)).cuda()
    out = torch.empty(max(1, int(np.prod(out_dims))), dtype=torch.int8, device="cuda")
    cap = max([1] + list(out_dims))
    rs = torch.empty(cap, dtype=torch.float32, device="cuda")
    rz = torch.empty(cap, dtype=torch.int32, device="cuda")
    rqd = hf.quant_broadcast_in_dim(x, dims, _qdev(q), bdims, out, out_dims, rs, rz, in_m2m=in_m2m, out_m2m=out_m2m)
    torch.cuda.synchronize()
    n = 1 if rqd < 0 else out_dims[rqd]
    return out.cpu().numpy()[: int(np.prod(out_dims))], rqd, rs.cpu().numpy()[:n], rz.cpu().numpy()[:n]


@pytest.mark.parametrize("seed", range(8))
def test_quant_broadcast_in_dim_vs_oracle(seed):
    """Random ranks, broadcast dimensions (some of size 1), layouts and quantization axes, per-axis and
    per-tensor: codes bit-exact, parameters equal to the oracle's (constraints C1, C6)."""
    g = np.random.default_rng(100 + seed)
    rank_in = int(g.integers(1, 4))
    rank_out = rank_in + int(g.integers(0, 3))
    bdims = g.choice(rank_out, size=rank_in, replace=False).tolist()
    out_dims = [int(v) for v in g.integers(1, 40, size=rank_out)]
    dims = [1 if g.random() < 0.3 else out_dims[b] for b in bdims]
    qd = int(g.integers(0, rank_in))
    if seed % 3 == 2:
        q = {"scales": np.float32([0.07]), "zero_points": np.int32([-5]), "quantization_dimension": None}
    else:
        q = {"scales": g.uniform(0.01, 0.5, dims[qd]).astype(np.float32),
             "zero_points": g.integers(-20, 21, dims[qd]).astype(np.int32), "quantization_dimension": qd}
    codes = g.integers(-128, 128, size=dims).astype(np.int8)
    in_m2m, out_m2m = g.permutation(rank_in).tolist(), g.permutation(rank_out).tolist()
    phys = _to_physical(codes, in_m2m)
    ref, params = oracle.quant_broadcast_in_dim(phys, dims, q, bdims, out_dims, m2m=in_m2m, out_m2m=out_m2m)
    got, rqd, rs, rz = _gpu_quant_broadcast(phys, dims, q, bdims, out_dims, in_m2m, out_m2m)
    assert np.array_equal(got, ref)
    assert rqd == (-1 if params["quantization_dimension"] is None else params["quantization_dimension"])
    assert np.array_equal(rs.view(np.uint32), params["scales"].view(np.uint32))
    assert np.array_equal(rz, params["zero_points"])


def test_quant_broadcast_in_dim_large_per_axis():
    """A per-axis vector s8[4096] (axis 0) broadcast to s8[4096, 4096] along dimension 1, column-major."""
    g = np.random.default_rng(5)
    n = 4096
    q = {"scales": g.uniform(0.001, 0.1, n).astype(np.float32), "zero_points": g.integers(-20, 21, n).astype(np.int32),
         "quantization_dimension": 0}
    codes = g.integers(-128, 128, size=n).astype(np.int8)
    ref, params = oracle.quant_broadcast_in_dim(codes, [n], q, [1], [n, n], out_m2m=[0, 1])
    got, rqd, rs, rz = _gpu_quant_broadcast(codes, [n], q, [1], [n, n], [0], [0, 1])
    assert np.array_equal(got, ref) and rqd == 1
    assert np.array_equal(rs, params["scales"]) and np.array_equal(rz, params["zero_points"])


@pytest.mark.parametrize("dtype", ["s8", "bf16", "f32"])
def test_reshape_layouts_vs_oracle(dtype):
    g = np.random.default_rng(11)
    cases = [([3, 4, 5], [6, 10]), ([8, 9, 10], [2, 4, 90]), ([1000, 33], [33, 1000]), ([7], [7, 1, 1])]
    npt = {"s8": np.int8, "bf16": np.uint16, "f32": np.float32}[dtype]
    for dims, out_dims in cases:
        x = g.integers(-100, 100, size=dims).astype(npt)
        for in_m2m in [list(range(len(dims) - 1, -1, -1)), list(range(len(dims)))]:
            for out_m2m in [list(range(len(out_dims) - 1, -1, -1)), list(range(len(out_dims)))]:
                phys = _to_physical(x, in_m2m)
                ref = oracle.reshape(phys, dims, out_dims, dtype, m2m=in_m2m, out_m2m=out_m2m)
                xt = torch.from_numpy(np.ascontiguousarray(phys).view({"s8": np.int8, "bf16": np.int16,
                                                                       "f32": np.float32}[dtype])).cuda()
                out = torch.empty_like(xt)
                hf.reshape(xt, dims, out, out_dims, dtype, in_m2m=in_m2m, out_m2m=out_m2m)
                torch.cuda.synchronize()
                got = out.cpu().numpy().view(npt)
                assert np.array_equal(got, ref), (dims, out_dims, in_m2m, out_m2m)


def test_quant_reshape_per_axis_keeps_parameters():
    """t[4, 3, 2] per-axis along 1 (the quantization page's example) reshaped to [2, 2, 3, 2] along 2: the
    codes move as the oracle moves them, in a non-default layout too."""
    g = np.random.default_rng(12)
    q = {"scales": np.float32([0.2, 0.1, 0.3]), "zero_points": np.int32([20, 10, 30]), "quantization_dimension": 1}
    codes = g.integers(-128, 128, size=[4, 3, 2]).astype(np.int8)
    for in_m2m, out_m2m in [([2, 1, 0], [3, 2, 1, 0]), ([0, 2, 1], [1, 3, 0, 2])]:
        phys = _to_physical(codes, in_m2m)
        ref = oracle.reshape(phys, [4, 3, 2], [2, 2, 3, 2], "s8", m2m=in_m2m, out_m2m=out_m2m, q=q, result_qdim=2)
        xt = torch.from_numpy(phys).cuda()
        out = torch.empty_like(xt)
        hf.reshape(xt, [4, 3, 2], out, [2, 2, 3, 2], "s8", q=_qdev(q), result_qdim=2, in_m2m=in_m2m, out_m2m=out_m2m)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), ref)
