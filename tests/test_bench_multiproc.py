"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks, each a replica with its own time and
byte count; rank 0 must see the max of the times and the sum of the bytes (weak scaling, no data-path
collective)."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    t = bench.aggregate(1.0 + rank, "max")      # replica times 1 s and 2 s
    b = bench.aggregate(100.0 * (rank + 1), "sum")  # bytes 100 and 200
    results[rank] = (t, b)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        out = dict(results)
    assert out[0] == (2.0, 300.0) and out[1] == (2.0, 300.0)


def test_single_process_aggregate_is_identity():
    import bench

    assert bench.aggregate(3.5, "max") == 3.5
    assert bench.aggregate(7.0, "sum") == 7.0


def test_gpus_flag_needs_one_process_per_gpu():
    """--gpus N > 1 without torchrun (WORLD_SIZE unset) is refused instead of silently running one replica."""
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--steps", "1"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 2
    assert "torch.distributed.run" in r.stderr


def test_fusion_kw_parsing():
    import bench

    assert bench.parse_kw("n=6144,dims=(3,512,2048)") == {"n": 6144, "dims": (3, 512, 2048)}
    assert bench.parse_kw("") == {}
