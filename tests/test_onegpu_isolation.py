"""Where the TMA multicast load may live (no GPU needed).

The library every process loads (libtmap_gb300.so), the benchmark and the build/smoke entry hold
no cluster-multicast TMA load: a multicast copy belongs only in code that one-GPU runs use alone.
It lives in the opt-in one-GPU library (async_bulk_tensor_tmap_gb300/onegpu), which the default
build does not compile and nothing but its own module and tests loads.
"""
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "async_bulk_tensor_tmap_gb300")
def _files(top, exts):
    for d, _, names in os.walk(top):
        if "_build" in d or "__pycache__" in d:
            continue
        for n in names:
            if n.endswith(exts):
                yield os.path.join(d, n)


def _holds_multicast_copy(path):
    src = open(path, encoding="utf-8", errors="replace").read()
    # a multicast TMA copy: a cp.async.bulk instruction string carrying .multicast::cluster
    return bool(re.search(r"cp\.async\.bulk[^;]*\.multicast::cluster", src.replace("\"\n", "").replace("\"", "")))


def test_multicast_copies_only_in_the_one_gpu_target():
    """Every compiled source of the repository (CUDA and C++ files) is searched for an inline-PTX
    bulk copy carrying .multicast::cluster."""
    onegpu = os.path.join(PKG, "onegpu")
    holders = [p for p in _files(ROOT, (".cu", ".cuh", ".cpp", ".cc"))
               if "_work" not in p and "baseline" not in p and _holds_multicast_copy(p)]
    assert holders, "the one-GPU target should hold the multicast load"
    assert all(p.startswith(onegpu + os.sep) for p in holders), holders


def test_default_build_bench_and_smoke_never_touch_the_one_gpu_target():
    build = open(os.path.join(PKG, "csrc", "build.py")).read()
    assert "onegpu" not in build and "k_gemm_multicast" not in build
    for f in ("bench.py", "__graft_entry__.py"):
        assert "onegpu" not in open(os.path.join(ROOT, f)).read(), f
    init = open(os.path.join(PKG, "__init__.py")).read()
    assert "onegpu" not in init


def test_one_gpu_library_builds_and_exports_its_calls():
    r = subprocess.run([sys.executable, os.path.join(PKG, "onegpu", "build.py")],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lib = r.stdout.strip().splitlines()[-1]
    syms = subprocess.run(["nm", "-D", "--defined-only", lib], capture_output=True, text=True).stdout
    header = open(os.path.join(ROOT, "include", "tmap_onegpu.h")).read()
    declared = re.findall(r"^(?:int|const char\*)\s+(\w+)\(", header, flags=re.M)
    assert set(declared) == {"stream_gemm_multicast", "tm_onegpu_check", "tm_onegpu_last_error"}
    for name in declared:
        assert re.search(rf"\bT {name}\b", syms), name
