"""Build libtmap_gb300_onegpu.so (sm_103a), the one-GPU-only companion library (see
include/tmap_onegpu.h).  Only on request: the package's default build never runs this, and no
benchmark or multi-GPU command loads the result."""
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
PKG = os.path.dirname(HERE)
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
SRC = os.path.join(HERE, "k_gemm_multicast.cu")
LIB = os.path.join(HERE, "libtmap_gb300_onegpu.so")
DEPS = [SRC, os.path.join(INCLUDE, "tmap.h"), os.path.join(INCLUDE, "tmap_onegpu.h")] + [
    os.path.join(CSRC, h) for h in ("tm_gemm.cuh", "tm_ptx.cuh", "tm_internal.h")]


def build(force: bool = False) -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        raise RuntimeError("nvcc not found; the one-GPU library cannot be built")
    if not force and os.path.exists(LIB) and all(os.path.getmtime(d) <= os.path.getmtime(LIB) for d in DEPS):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC,
           SRC, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
