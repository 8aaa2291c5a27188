"""hlo_reduce_fusion_noalloc: the reduce entry point that allocates no device memory.

Some callers cannot allocate device memory where they run a reduction (code embedded in a runtime that
owns all device memory through its own allocator, or held to a memory budget fixed at start-up), so
they cannot pass hlo_reduce_fusion a workspace. The no-allocation entry point keeps the split-row
partials in a fixed scratch array the library holds on the device. Here it is called through the C ABI
twice in a row on reductions that split their rows (and one that does not) and compared with
hlo_reduce_fusion given a workspace, within the reduction tolerance of the other tests.

The file is named so that pytest collects it last.
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import transpose_heroes_gb300 as hf
from transpose_heroes_gb300 import inputs as inp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transpose_heroes_gb300 import build

    build.build()
    oracle.build()
    hf.lib()


# (dims, dtype, kind, init, prologue): the first three split their rows, the last does not
CASES = [
    ([1, 1 << 22], "f32", "add", 0.0, ["exp"]),
    ([3, 1000003], "f32", "max", -math.inf, None),
    ([10, 1 << 20], "bf16", "add", 2.5, ["exp"]),
    ([4096, 512], "f32", "add", 0.0, ["exp"]),
]


def _tolerance(data, dims, dtype, kind, init, ops):
    """The reduction tolerance of the parity tests: 1e-5 * sum|terms| + 1e-6 (add), exact (max)."""
    if kind == "max":
        return np.zeros(dims[0])
    _, asum = oracle.reduce(data, dims, dtype, [1], kind, init, "f32",
                            prologue={"ops": ops, "round_each": True} if ops else None, want_abs_sum=True)
    return 1e-5 * asum + 1e-6


@pytest.mark.parametrize("case", range(len(CASES)))
def test_noalloc_reduce_matches_the_workspace_entry_point(case):
    dims, dtype, kind, init, ops = CASES[case]
    g = inp.rng(case + 1)
    n = int(np.prod(dims))
    data = inp.uniform_f32(g, n, -1, 1) if dtype == "f32" else inp.normal_bf16(g, n)
    x = torch.from_numpy(data.view(np.int16) if dtype == "bf16" else data).cuda()
    pro = {"ops": ops, "round_each": True} if ops else None
    ws_bytes = hf.reduce_workspace_size(dims, dtype, [1])
    assert (ws_bytes > 0) == (case < 3)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    ref = torch.empty(dims[0], dtype=torch.float32, device="cuda")
    hf.reduce_fusion(x, dims, dtype, [1], kind, init, ref, "f32", prologue=pro, workspace=ws if ws_bytes else None,
                     workspace_bytes=ws_bytes)
    tol = _tolerance(data, dims, dtype, kind, init, ops)
    for _ in range(2):  # two calls in a row: the second finds the first one's partials in the scratch
        out = torch.full((dims[0],), float("nan"), dtype=torch.float32, device="cuda")
        hf.reduce_fusion_noalloc(x, dims, dtype, [1], kind, init, out, "f32", prologue=pro)
        torch.cuda.synchronize()
        got, want = out.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
        err = np.abs(got - want)
        assert np.all(err <= tol), f"worst error {err.max()} against tolerance {tol[np.argmax(err)]}"
