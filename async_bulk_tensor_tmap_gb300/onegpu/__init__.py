"""One-GPU-only companion of the library: the tensor-core GEMM with its B tile shared by the two
CTAs of a cluster through TMA multicast (include/tmap_onegpu.h).  Argument marshalling only.

Importing this module is the opt-in: it builds libtmap_gb300_onegpu.so if needed and loads it.
The package's default build, bench.py and every multi-GPU command never import it, so no process
of a multi-GPU run holds a multicast load; the library itself refuses tensors that are not device
memory of the current device, and refuses to run in one rank of several (WORLD_SIZE > 1).

    stream_gemm_multicast(a, b_half, c, ldc=None, stages=4, stream=None)
        a: TensorMap {K, M}, box {64, 128}; b_half: TensorMap {K, N} of B, box {64, 128};
        c: fp32 device tensor (M x N, row stride ldc, default N)
    tm_onegpu_check(stream=None)

    python -m async_bulk_tensor_tmap_gb300.onegpu [M N K]   times it against stream_gemm
"""
from __future__ import annotations

import ctypes
import os

from .. import TM_OK, TmapError
from .build import build

if int(os.environ.get("WORLD_SIZE", "1")) > 1:
    raise ImportError("async_bulk_tensor_tmap_gb300.onegpu is for one-GPU processes only")

library_path = build()
_L = ctypes.CDLL(library_path)
_vp = ctypes.c_void_p
_L.stream_gemm_multicast.argtypes = [_vp, _vp, _vp, ctypes.c_uint64, ctypes.c_uint32, _vp]
_L.stream_gemm_multicast.restype = ctypes.c_int
_L.tm_onegpu_check.argtypes = [_vp]
_L.tm_onegpu_check.restype = ctypes.c_int
_L.tm_onegpu_last_error.restype = ctypes.c_char_p


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    return stream if isinstance(stream, int) else int(stream.cuda_stream)


class OneGpuError(TmapError):
    """A non-zero status of this library (its own last-error text)."""

    def __init__(self, code: int, where: str):
        RuntimeError.__init__(self, f"{where} failed with status {code}: "
                                    f"{_L.tm_onegpu_last_error().decode(errors='replace')}")
        self.code = code


def _check(rc: int, what: str) -> None:
    if rc != TM_OK:
        raise OneGpuError(rc, what)


def stream_gemm_multicast(a, b_half, c, ldc=None, stages: int = 4, stream=None) -> None:
    n = b_half.dims[1]
    _check(_L.stream_gemm_multicast(a.ptr, b_half.ptr, c.data_ptr(), n if ldc is None else ldc,
                                    stages, _stream(stream)), "stream_gemm_multicast")


def tm_onegpu_check(stream=None) -> int:
    return int(_L.tm_onegpu_check(_stream(stream)))


def last_error() -> str:
    return _L.tm_onegpu_last_error().decode()
