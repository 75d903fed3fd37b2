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


class _FakeSmi:
    """Stands in for the nvidia-smi process: canned CSV lines."""

    def __init__(self, text):
        self.text = text

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.text, ""


def test_clock_sampler_uses_samples_inside_the_timed_region():
    import datetime
    sys.path.insert(0, ROOT)
    import bench
    t0 = datetime.datetime(2026, 12, 2, 9, 0, 0)
    lines = []
    for i in range(10):  # every 100 ms; the region spans samples 3..6
        t = t0 + datetime.timedelta(milliseconds=100 * i)
        busy = 3 <= i <= 6
        lines.append(", ".join([t.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3], "0",
                                "1850" if busy else "2070", "2070", "1300.5" if busy else "200.0", "0",
                                "0x4" if busy else "0x0", "Not Active", "Not Active", "Not Active",
                                "Active" if busy else "Not Active"]))
    s = bench.ClockSampler(0)
    s.proc = _FakeSmi("\n".join(lines))
    s.window = (t0 + datetime.timedelta(milliseconds=250), t0 + datetime.timedelta(milliseconds=650))
    c = s.stop()
    assert c["samples"] == 10 and c["samples_under_load"] == 4
    assert c["sm_mhz"] == 1850 and c["sm_max_mhz"] == 2070 and c["reasons"] == ["sw_power_cap"]
    assert c["power_w_median"] == 1300.5
    # no window (or none inside it): every sample is used and said so
    s = bench.ClockSampler(0)
    s.proc = _FakeSmi("\n".join(lines))
    c = s.stop()
    assert c["samples_under_load"] == 0 and c["selection"].startswith("all samples")
