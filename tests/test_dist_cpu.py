"""Multi-rank bookkeeping of bench.py on CPU (gloo, world size 2).

Decode sequences are independent, so ranks run replicas with no collective on
the data path; the only cross-rank steps are the barrier and the max of the
elapsed times, which these tests exercise without a GPU."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        dist.barrier()
        mine = 10.0 + 5.0 * rank  # rank 1 is the slower one
        worst = bench.max_over_ranks(mine, torch.device("cpu"))
        ws, r, _ = bench.dist_env()
        results[rank] = (worst, ws, r, bench.job_throughput(ws, 1_000_000, worst))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_two_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(results)
    assert res[0][0] == res[1][0] == 15.0
    assert (res[0][1], res[0][2], res[1][2]) == (2, 0, 1)
    # 2 ranks x 1 MB per step in 15 ms
    assert res[0][3] == pytest.approx(2 * 1e6 / 15e-3 / 1e9)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
    assert bench.job_throughput(1, 4_000_000_000, 1000.0) == pytest.approx(4.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    """`bench.py --impl reference` launched by torchrun with two ranks on the
    CPU: rank 0 alone runs the oracle and prints one JSON line, rank 1 exits 0
    without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3", "--ref-seqs", "2"]
    res = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
