"""The multi-rank bench path on the CPU: two gloo ranks aggregate their
timings the way bench.py does under torchrun (slowest rank's time, all
ranks' bytes; weak scaling, no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    seconds = 0.5 + rank  # rank 1 is the slowest
    slowest, value = bench.aggregate(seconds, 1_000_000, 10, dist, "cpu")
    out[rank] = torch.tensor([slowest, value], dtype=torch.float64)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    out = torch.zeros(world, 2, dtype=torch.float64).share_memory_()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    # both ranks see the slowest rank's time and the whole job's bytes
    for r in range(world):
        assert out[r, 0].item() == pytest.approx(1.5)
        assert out[r, 1].item() == pytest.approx(1_000_000 * 10 * world / 1.5 / 1e9)


def test_single_rank_aggregation():
    import bench
    slowest, value = bench.aggregate(2.0, 4e9, 3)
    assert slowest == 2.0 and value == pytest.approx(4e9 * 3 / 2.0 / 1e9)


def test_reference_arm_under_two_ranks():
    """torchrun with two ranks: rank 0 times the oracle and prints one JSON
    line; rank 1 exits 0 without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
