"""Host-side checks of bench.py (no GPU): the multi-replica aggregation over
two gloo ranks, and the reference arm's JSON line on a tiny budget."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r pretends its timed region took (r + 1) seconds for 10 steps of 3 units
        t, rate = bench.aggregate(float(rank + 1), 3.0, 10, dist, "cpu")
        out.put((rank, t, rate))
    finally:
        dist.destroy_process_group()


def test_replicas_take_max_time_and_sum_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest rank's 2 s and the work of both replicas
    assert [(r, t) for r, t, _ in got] == [(0, 2.0), (1, 2.0)]
    assert all(rate == pytest.approx(2 * 3.0 * 10 / 2.0) for _, _, rate in got)


def test_single_process_aggregate():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(0.5, 4.0, 100) == (0.5, 800.0)


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--shape", "square512", "--steps", "3", "--warmup", "3",
                          "--ref-budget", "1"], capture_output=True, text=True, timeout=300,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["steps"] == 3


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3"], capture_output=True, text=True,
                         timeout=120, cwd=ROOT, env=env)
    assert out.returncode == 0 and out.stdout.strip() == ""
