"""The multi-process side of bench.py on the CPU: two gloo ranks (127.0.0.1).

bench.py --gpus N runs N independent replicas (one per GPU); the job's time
is the slowest rank's and the value counts every rank's tokens.  The
reduction and the value are tested here with two processes; the reference
arm is launched under torchrun with two ranks to check that only rank 0
works and prints, and that every rank exits 0."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank r took (10 + r) ms for the main line and (30 - r) ms end to end
        got = bench.max_over_ranks([10.0 + rank, 30.0 - rank])
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    # every rank holds the slowest rank's time of each figure
    assert res[0] == [11.0, 30.0] and res[1] == [11.0, 30.0]


def test_max_over_ranks_is_identity_without_a_group():
    assert bench.max_over_ranks([3.5, 1.25]) == [3.5, 1.25]


def test_job_value_counts_every_rank():
    # 2 ranks x 1 token x 100 steps in 250 ms -> 800 tokens/s
    assert bench.job_tokens_per_s(2, 1, 100, 250.0) == pytest.approx(800.0)
    assert bench.job_tokens_per_s(1, 4096, 1, 8.0) == pytest.approx(512000.0)


def test_reference_arm_under_torchrun_prints_once_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1", "--workload", "tiny"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
