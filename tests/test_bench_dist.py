"""The N > 1 path of bench.py on CPU (gloo, world size 2): replicas only, so
the only collectives are the timing barrier and the max over ranks; rank 0
alone prints, with the whole-job aggregate."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, port: int, q):
    import torch

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                      LOCAL_RANK=str(rank))
    dist, r, world, local = bench._dist()
    bench._DIST = dist
    bench._barrier()
    mx = bench._max_over_ranks(10.0 + 5.0 * rank, torch.device("cpu"))  # rank 1 is the slow one
    q.put((r, world, local, mx, bench.whole_job_gbs(1e9, world, mx, 4)))
    bench._barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1] and all(o[1] == 2 for o in out)
    assert all(o[3] == 15.0 for o in out)                    # both ranks see the slowest rank's time
    assert all(abs(o[4] - 2e9 / (15.0 / 4) / 1e6) < 1e-6 for o in out)  # both ranks' bytes over the max


def test_whole_job_aggregate():
    assert bench.whole_job_gbs(1.6e9, 1, 3.2, 10) == pytest.approx(1.6e9 / 0.32e-3 / 1e9)
    assert bench.whole_job_gbs(1.6e9, 4, 3.2, 10) == pytest.approx(4 * bench.whole_job_gbs(1.6e9, 1, 3.2, 10))


def test_reference_arm_under_torchrun_prints_once():
    """A torch.distributed.run launch with two ranks, on CPU: rank 0 alone prints one line."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "1", "--cpu-budget", "0.5"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
