"""bench.py's reference arm (the oracle timed on the host cores) on the CPU:
the JSON line carries the contract's keys, its value is the cpu_baseline's
and the e2e's, and the sample it describes is what the oracle processed."""
from __future__ import annotations

import json
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_reference(workload, steps=2, warmup=1):
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", workload, "--steps", str(steps), "--warmup", str(warmup)],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("workload, tokens", [("gdn_fp32_t256", 256)])
def test_reference_line(workload, tokens):
    d = run_reference(workload)
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["config"]["workload"] == workload
    assert d["higher_is_better"] is True and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    # the sample names a token count no larger than the workload, and the
    # value is that count over the step time
    n = int(re.search(r"first (\d+) tokens", cb["sample"]).group(1))
    assert 1 <= n <= tokens
    assert d["value"] == pytest.approx(n / (d["ms_per_step"] / 1e3), rel=1e-9)


def test_sample_text_names_rows_and_sequences():
    import torch

    sys.path.insert(0, ROOT)
    import bench

    class C:
        HV, name = 4, "w"

    one = {"q": torch.empty(1, 10, 1, 1), "cu_seqlens": None}
    two = {"q": torch.empty(2, 10, 1, 1), "cu_seqlens": None}
    packed = {"q": torch.empty(1, 10, 1, 1), "cu_seqlens": torch.tensor([0, 3, 10])}
    assert "first 7 tokens (all 4" in bench.oracle_sample_text(C, one, 7)
    assert "first 5 tokens of each of the 2 batch rows (10 tokens)" in \
        bench.oracle_sample_text(C, two, 10)
    assert "first 3 tokens of the first packed sequence" in \
        bench.oracle_sample_text(C, packed, 3)
