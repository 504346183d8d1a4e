"""bench.py's GPU arm on a small scale: one JSON line with every key of the contract (roofline of
the dominant kernel, the end-to-end leg with its host bytes, the SM clock record and the count of
library launches; cpu_baseline and the recorded DRAM traffic belong to the full-size workload and
are null here), its values consistent with each other."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_gpu_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3",
                        "--warmup", "3", "--scale", "8", "--e2e-steps", "2"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "e2e", "cpu_baseline", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["warmup"] >= 3 and d["value"] > 0
    rf = d["roofline"]
    assert rf["bound"] in ("hbm", "tensor", "alu") and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert rf["traffic"] is None  # the recorded traffic is for the full-size launch only
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["cpu_baseline"] is None  # reported for the full-size workload only
    assert d["gpu_launches"] == len(d["breakdown"]) * d["steps"]
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
