"""bench.py's reference arm on CPU (it times the oracle on the host cores): one JSON line carrying
the contract's keys, with the metric, unit and direction of the GPU arm, an e2e object that moves
no bytes, and a cpu_baseline that describes the run."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1", "--scale", "32"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e",
              "cpu_baseline"):
        assert k in d, k
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert "workload" in d["config"]


def test_recorded_traffic_follows_the_kernel_code(tmp_path, monkeypatch):
    """bench.py reports a recorded DRAM traffic only while the streaming kernel's code is the one
    it was captured on: a comment or blank-line edit keeps it, a code edit voids it."""
    import hashlib
    import shutil
    sys.path.insert(0, ROOT)
    import bench
    csrc = os.path.join("async_bulk_tensor_tmap_gb300", "csrc")
    os.makedirs(tmp_path / csrc)
    os.makedirs(tmp_path / "profiles")
    for f in ("k_tma.cu", "tm_ptx.cuh", "tm_internal.h"):
        shutil.copy(os.path.join(ROOT, csrc, f), tmp_path / csrc / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    digest = hashlib.sha256(bench.tma_kernel_source()).hexdigest()
    (tmp_path / "profiles" / "roofline_traffic.txt").write_text(
        f"# a record\nkernel: w5a.reduce\nsource_sha256: {digest}\ntraffic_bytes: 123\n")
    assert bench.recorded_traffic("w5a.reduce") == 123
    assert bench.recorded_traffic("w3.copy") is None
    k = tmp_path / csrc / "k_tma.cu"
    src = k.read_text()
    k.write_text("// a note\n\n" + src.replace("\n", "  // x\n", 3))
    assert bench.recorded_traffic("w5a.reduce") == 123
    k.write_text(src.replace("{", "{ ;", 1))
    assert bench.recorded_traffic("w5a.reduce") is None
