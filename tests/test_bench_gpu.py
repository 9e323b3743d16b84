"""The bench's JSON line on the GPU: one short run of the default workload
through bench.py, as it is launched at N = 1, checked for the keys of its
contract (the metric and its value, the kernel roofline against a measured or
fallback peak, the oracle's CPU baseline, the end-to-end rate with the bytes it
copies, the clocks sampled during the timed region, the launch count)."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_default_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3",
                          "--warmup", "3", "--e2e-steps", "2", "--cpu-seconds", "1"],
                         capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["warmup"] == 3
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "gdn_bf16_t32768"
    r = line["roofline"]
    assert r["bound"] in ("hbm", "tensor") and r["peak"] > 0 and 0 < r["frac"] < 1.5
    assert r["achieved"] == pytest.approx(r["frac"] * r["peak"], rel=1e-6)
    e = line["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    c = line["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0
    assert line["gpu_launches"] > 0
    assert "sm_mhz" in line["clocks"] and "reasons" in line["clocks"]
    # the single-call and lockstep rates of the same workload
    assert line["single_call"]["ms_per_step"] > 0 and line["lockstep"]["ms_per_step"] > 0
