"""Host-side arithmetic of bench.py (CPU only): the algorithmic bytes and
FLOPs the roofline fraction divides by, and the clock sampler's restriction
to the timed region."""
import time

import numpy as np
import pytest

import bench
from sink_sda_decode_gb300 import inputs


class _W:
    """Just the fields the formulas read."""

    def __init__(self, N, H, D, total_len):
        self.N, self.H, self.D, self.total_len = N, H, D, total_len


def test_algorithmic_bytes_and_flops_match_the_published_config_figures():
    # N=64, H=16, D=512, 640 slots per token: 44.20 MB and 1.342 GFLOP
    w = _W(64, 16, 512, 64 * 640)
    b = bench.algorithmic_bytes(w)
    assert b == 40960 * 1024 + 2 * 64 * 16 * 512 * 2 + 40960 * 4 + 65 * 4
    assert abs(b / 1e6 - 44.20) < 0.01
    assert bench.algorithmic_flops(w) == 4 * 16 * 512 * 40960
    assert abs(bench.algorithmic_flops(w) / 1e9 - 1.342) < 0.001
    # N=1024, H=128, L=640: 942.15 MB and 171.8 GFLOP
    w = _W(1024, 128, 512, 1024 * 640)
    assert abs(bench.algorithmic_bytes(w) / 1e6 - 942.15) < 0.01
    assert abs(bench.algorithmic_flops(w) / 1e9 - 171.8) < 0.05


def test_fp8_pool_bytes():
    # an FP8 row is D one-byte codes plus a 4-byte scale
    w = _W(64, 16, 512, 64 * 640)
    assert bench.algorithmic_bytes(w, "fp8") == 40960 * (512 + 4) + 2 * 64 * 16 * 512 * 2 + 40960 * 4 + 65 * 4
    assert bench.algorithmic_bytes(w, "fp8") < bench.algorithmic_bytes(w)


def test_bytes_follow_the_generated_workload():
    w = inputs.config(0)  # the tiny case: lengths {0, 1, 17, 64}
    assert int(w.total_len) == 82
    assert bench.algorithmic_bytes(w) == 82 * w.D * 2 + 2 * w.N * w.H * w.D * 2 + 82 * 4 + (w.N + 1) * 4


def test_clock_summary_keeps_only_samples_inside_the_timed_region():
    cs = bench.ClockSampler(0)
    cs.max_mhz, cs.source = 2070.0, "test"
    t = time.perf_counter()
    cs.samples = [(t - 1.0, 345.0, {"hw_slowdown"}),      # before: idle clock, must not count
                  (t + 0.1, 2070.0, set()),
                  (t + 0.2, 2040.0, {"sw_power_cap"}),
                  (t + 5.0, 900.0, {"sw_thermal_slowdown"})]  # after
    cs.mark(t, t + 1.0)
    s = cs.summary()
    assert s["samples"] == 2
    assert s["sm_mhz"] == pytest.approx(2055.0)
    assert s["reasons"] == ["sw_power_cap"]
    assert s["sm_max_mhz"] == 2070.0


def test_kernel_source_hash_is_stable_and_short():
    h = bench.kernel_source_hash()
    assert h == bench.kernel_source_hash() and len(h) == 16
    int(h, 16)


def test_store_bytes_by_hand():
    # H=16, D=512, R=64: q read + written 2*16*512*2, KV row read 1024 and
    # stored 1024 (FP8: 512 codes + 4-byte scale), 8 bytes of slot/position,
    # 64*4 bytes of cos/sin, plus the two 1 KB weights once
    w = _W(64, 16, 512, 0)
    per = 2 * 16 * 512 * 2 + 1024 + 1024 + 8 + 256
    assert bench.store_algorithmic_bytes(w, 64) == 64 * per + 2048
    assert bench.store_algorithmic_bytes(w, 64, "fp8") == 64 * (per - 1024 + 516) + 2048


def test_topk_bytes_by_hand():
    # lengths 0, 100, 8192 with k=512, K=64: scores 4 B each, lengths 4 B,
    # block-table rows ceil(n/64)*4 B, indptr (N+1)*4 B, 8 B per kept position
    b = bench.topk_algorithmic_bytes([0, 100, 8192], 512, 64)
    assert b == (0 + 100 + 8192) * 4 + 3 * 4 + (0 + 2 + 128) * 4 + 4 * 4 + (0 + 100 + 512) * 8


def test_kernel_source_hashes_cover_each_measured_kernel():
    hs = {k: bench.kernel_source_hash(k) for k in ("decode", "store", "topk")}
    assert len(set(hs.values())) == 3 and all(len(h) == 16 for h in hs.values())
    assert bench.ncu_traffic("no such workload") is None


@pytest.mark.parametrize("path,metric", [("store", bench.STORE_METRIC), ("topk", bench.TOPK_METRIC),
                                         ("layer", bench.METRIC)])
def test_reference_arm_of_every_path(path, metric):
    """`bench.py --impl reference --path P` times the oracle's share of that
    path's step on the CPU and prints one line with the path's metric."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.abspath(bench.__file__))
    cmd = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--path", path,
           "--config", "h16", "--steps", "1", "--warmup", "1"]
    p = subprocess.run(cmd, cwd=root, env=dict(os.environ, OMP_NUM_THREADS="2"),
                       capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["metric"] == metric and line["value"] > 0
    assert line["config"]["path"] == path


@pytest.mark.parametrize("path", ["decode", "store", "topk", "layer"])
def test_report_line_of_every_path(path):
    """The JSON line each path prints: its metric, the byte count its
    roofline divides by, its launch count and the keys the contract asks for."""
    class Args:
        steps, warmup, config, kv = 10, 3, "h16", "bf16"
    Args.path = path
    w = inputs.config(1)
    ti_bytes = 1234567
    r = {"h2d": 10, "d2h": 20, "clocks": {"sm_mhz": 2070.0}, "rope_dim": 64,
         "topk_bytes": ti_bytes, "launches_per_step": {"decode": 5, "store": 1, "topk": 2,
                                                       "layer": 6}[path]}
    line = bench.report_line(Args, w, 1, 0.040, 0.020, 0.060, w.N, r)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in line
    rf = line["roofline"]
    assert rf["bound"] == "hbm" and rf["kernel_ms"] == 0.020
    want = {"store": bench.store_algorithmic_bytes(w, 64), "topk": ti_bytes}.get(
        path, bench.algorithmic_bytes(w))
    assert rf["algorithmic_bytes"] == want
    assert rf["achieved"] == pytest.approx(want / 1e9 / 20e-6)
    assert line["gpu_launches"] == r["launches_per_step"] * 10
    assert line["metric"] == {"store": bench.STORE_METRIC, "topk": bench.TOPK_METRIC}.get(path, bench.METRIC)
    assert line["value"] == pytest.approx(w.N / 40e-6) and line["e2e"]["value"] == pytest.approx(w.N / 60e-6)
    assert line["config"]["path"] == path


def test_distinct_row_bytes():
    """Each distinct pool row counted once: equal to the algorithmic bytes
    when no row repeats, smaller by the repeats' row bytes otherwise."""
    w = inputs.random_small(3, 6, 4, 64, 1000, [7, 0, 3, 9, 1, 5])
    assert len(set(w.kv_indices.tolist())) == w.kv_indices.size
    assert bench.distinct_row_bytes(w) == bench.algorithmic_bytes(w)
    d = inputs.random_small(4, 6, 4, 64, 8, [7, 0, 3, 9, 1, 5], duplicates=True)
    repeats = d.kv_indices.size - len(set(d.kv_indices.tolist()))
    assert repeats > 0
    assert bench.distinct_row_bytes(d) == bench.algorithmic_bytes(d) - repeats * 64 * 2
    assert bench.distinct_row_bytes(d, "fp8") == bench.algorithmic_bytes(d, "fp8") - repeats * (64 + 4)


def test_report_line_distinct_rows():
    class Args:
        steps, warmup, config, kv, path = 10, 3, "h16", "bf16", "decode"
    w = inputs.config(1)
    r = {"h2d": 10, "d2h": 20, "clocks": {"sm_mhz": 2070.0}, "launches_per_step": 5}
    rf = bench.report_line(Args, w, 1, 0.040, 0.020, 0.060, w.N, r)["roofline"]
    assert rf["distinct_row_bytes"] == bench.distinct_row_bytes(w) <= rf["algorithmic_bytes"]
    assert rf["frac_distinct_rows"] == pytest.approx(rf["distinct_row_bytes"] / 1e9 / 20e-6 / rf["peak"])
