"""Build libtmap_gb300.so (sm_103a) in-tree with nvcc: one object per source, compiled in
parallel, linked with the static CUDA runtime (no link-time dependency on libcuda).

build(trace=True) builds the tracing variant instead, libtmap_gb300_trace.so (-DTM_TRACE: the
streaming kernels and the ring write a %globaltimer stamp per CTA at fixed points; see
async_bulk_tensor_tmap_gb300/timeline.py).  The default build never makes or loads it."""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

CSRC = os.path.dirname(os.path.abspath(__file__))
PKG = os.path.dirname(CSRC)
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtmap_gb300.so")
TRACE_LIB = os.path.join(PKG, "libtmap_gb300_trace.so")

SOURCES = ["tmap_host.cpp", "k_tma.cu", "k_fallback.cu", "k_fb_seg.cu", "k_ring.cu", "k_gemm.cu",
           "tm_noalloc.cu"]
HEADERS = ["tm_internal.h", "tm_ptx.cuh", "tm_gemm.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA library cannot be built")
    return cand


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), trace: bool = False) -> str:
    build_dir = os.path.join(BUILD, "trace") if trace else BUILD
    lib = TRACE_LIB if trace else LIB
    if trace:
        extra_flags = (*extra_flags, "-DTM_TRACE")
    os.makedirs(build_dir, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "tmap.h")]
    objs = []
    jobs = []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        objs.append(obj)
        if force or _stale(obj, [path] + hdrs):
            cmd = [nvcc(), *ARCH, *FLAGS, *extra_flags, "-c", path, "-o", obj]
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)

    with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else [],
                trace="--trace" in sys.argv))
