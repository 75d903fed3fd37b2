"""Host-side checks of bench.py (no GPU): the one-GPU rule, the compact
per-shape summary that ends the JSON line, and the reference arm's JSON line
on a tiny budget."""
from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_more_than_one_gpu_is_refused():
    for n in ("2", "8", "0"):
        out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", n],
                             capture_output=True, text=True, timeout=120, cwd=ROOT)
        assert out.returncode == 2 and out.stdout.strip() == ""
        assert "one GPU" in out.stderr


def test_single_process_aggregate():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(0.5, 4.0, 100) == (0.5, 800.0)


def test_compact_shape_summary():
    sys.path.insert(0, ROOT)
    import bench
    rec = {"us": 31.5, "roofline": {"frac": 0.6561, "bound": "hbm"}, "cublas_us": 29.4,
           "clocks": {"sm_mhz": 2017.0}, "median_us": 37.0, "kernel_config": {"grid": 128},
           "graph_us": 2347.16, "cublas_graph_us": 2287.07}
    assert bench.compact_shape(rec) == {"us": 31.5, "hbm": 0.6561, "cb_us": 29.4,
                                        "g_us": 2347.16, "cb_g_us": 2287.07, "mhz": 2017}
    # the longest values: a tensor-bound shape of a few milliseconds
    rec = dict(rec, us=2347.16, cublas_us=2287.07, roofline={"frac": 0.8599, "bound": "tensor"})
    # the twelve shapes besides the headline stay short enough for a
    # 1500-character tail of the output (the line is printed without spaces)
    line = json.dumps({name: bench.compact_shape(rec) for name in bench.EXTRA_SHAPES},
                      separators=(",", ":"))
    assert len(line) < 1300


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


def test_tensor_peak_regime_follows_the_timed_region():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.tensor_peak_regime(0.004) == "burst"
    assert bench.tensor_peak_regime(1.07) == "sustained"
    assert bench.tensor_peak_regime(bench.SUSTAINED_REGION_S) == "sustained"
