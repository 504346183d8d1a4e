"""Python binding of libtmap_gb300.so (see include/tmap.h): argument marshalling only.

Every operation runs in the library's CUDA kernels.  PyTorch supplies device memory and streams;
a tensor argument is only read for its data_ptr(), and `stream` defaults to torch's current
stream.  There is no CPU fallback: if the library was not built this module refuses to import.

Function names and argument order follow the C ABI:
    tmap_plan / tmap_encode(dtype, base, global_dim, global_strides, box_dim, element_strides=None,
                            swizzle=TM_SWIZZLE_NONE, oob=TM_OOB_ZERO) -> TensorMap
    tmap_replace_address(map, new_base), tmap_force_fallback(map), tmap_set_l2_promotion(map, promo)
    tile_load_image(src, coords, image, stream=None)
    tiled_copy(src, coords, images, stream=None)            coords None = whole box grid
    tiled_roundtrip(dst, coords, images, stream=None)
    tiled_copy_noalloc(src, coords, images, stream=None)  no device allocation, returns when done
    tile_reduce_add(dst, src, stream=None), tile_reduce(dst, src, op, stream=None)
    stream_tiles(a, b, stages, cs_a, cs_b, bits_a, bits_b, stream=None)
    tm_stream_check(stream=None), tm_selftest_wait_timeout(timeout_ns, stream=None)
Dimension lists are innermost first, as in the C ABI.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "TmapError", "TensorMap", "tmap_plan", "tmap_encode", "tmap_replace_address",
    "tmap_force_fallback", "tmap_set_l2_promotion", "TM_L2_NONE", "TM_L2_64B", "TM_L2_128B",
    "TM_L2_256B", "tile_load_image", "tiled_copy", "tiled_roundtrip", "tile_reduce_add",
    "tile_reduce", "TM_RED_ADD", "TM_RED_MIN", "TM_RED_MAX",
    "stream_tiles", "stream_gemm", "tiled_copy_noalloc", "TM_NOALLOC_MAX_BOXES", "tm_stream_check",
    "tm_selftest_wait_timeout", "tm_pick_swizzle", "tm_last_error",
    "library_path", "TM_OK", "TM_EINVAL", "TM_EALIGN", "TM_ERANGE", "TM_EUNSUPPORTED",
    "TM_ECUDA", "TM_ETIMEOUT", "TM_U8", "TM_U16", "TM_U32", "TM_S32", "TM_U64", "TM_S64",
    "TM_F16", "TM_F32", "TM_F64", "TM_BF16", "TM_SWIZZLE_NONE", "TM_SWIZZLE_32B",
    "TM_SWIZZLE_64B", "TM_SWIZZLE_128B", "TM_OOB_ZERO", "TM_OOB_NAN", "TM_PATH_TMA",
    "TM_PATH_FALLBACK", "TM_WHY_STRIDE", "TM_WHY_BASE", "TM_WHY_DRIVER", "TM_WHY_FORCED", "TM_WHY_STEP0",
]

TM_OK, TM_EINVAL, TM_EALIGN, TM_ERANGE, TM_EUNSUPPORTED, TM_ECUDA, TM_ETIMEOUT = range(7)
TM_U8, TM_U16, TM_U32, TM_S32, TM_U64, TM_S64, TM_F16, TM_F32, TM_F64, TM_BF16 = range(10)
TM_SWIZZLE_NONE, TM_SWIZZLE_32B, TM_SWIZZLE_64B, TM_SWIZZLE_128B = range(4)
TM_OOB_ZERO, TM_OOB_NAN = 0, 1
TM_PATH_TMA, TM_PATH_FALLBACK = 1, 2
TM_RED_ADD, TM_RED_MIN, TM_RED_MAX = 0, 1, 2
TM_WHY_STRIDE, TM_WHY_BASE, TM_WHY_DRIVER, TM_WHY_FORCED, TM_WHY_STEP0 = 1, 2, 4, 8, 16
TM_L2_NONE, TM_L2_64B, TM_L2_128B, TM_L2_256B = range(4)
DESC_SIZE = 384
TM_NOALLOC_MAX_BOXES = 16384

_HERE = os.path.dirname(os.path.abspath(__file__))
# TMAP_GB300_TRACE=1 loads the tracing build (per-CTA timelines, async_bulk_tensor_tmap_gb300.timeline)
_TRACE = os.environ.get("TMAP_GB300_TRACE") == "1"
library_path = os.path.join(_HERE, "libtmap_gb300_trace.so" if _TRACE else "libtmap_gb300.so")

if not os.path.exists(library_path):
    raise ImportError(
        f"{library_path} is missing: build the CUDA library first "
        "(python -c 'import __graft_entry__ as g; g.build()')")

_L = ctypes.CDLL(library_path)

_vp = ctypes.c_void_p
_u32, _u64, _i32 = ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int32
_P = ctypes.POINTER

_SIGS = {
    "tmap_plan": [_vp, ctypes.c_int, _u32, _vp, _P(_u64), _P(_u64), _P(_u32), _P(_u32),
                  ctypes.c_int, ctypes.c_int],
    "tmap_encode": [_vp, ctypes.c_int, _u32, _vp, _P(_u64), _P(_u64), _P(_u32), _P(_u32),
                    ctypes.c_int, ctypes.c_int],
    "tmap_replace_address": [_vp, _vp],
    "tmap_force_fallback": [_vp],
    "tmap_set_l2_promotion": [_vp, ctypes.c_int],
    "tile_load_image": [_vp, _P(_i32), _vp, _vp],
    "tiled_copy": [_vp, _P(_i32), ctypes.c_size_t, _vp, _vp],
    "tiled_roundtrip": [_vp, _P(_i32), ctypes.c_size_t, _vp, _vp],
    "tiled_copy_noalloc": [_vp, _P(_i32), ctypes.c_size_t, _vp, _vp],
    "tile_reduce_add": [_vp, _vp, _vp],
    "tile_reduce": [_vp, _vp, ctypes.c_int, _vp],
    "stream_tiles": [_vp, _vp, _u32, _vp, _vp, _vp, _vp, _vp],
    "stream_gemm": [_vp, _vp, _vp, _u64, _u32, _vp],
    "tm_stream_check": [_vp],
    "tm_selftest_wait_timeout": [_u64, _vp],
    "tm_last_error": [],
    "tm_box_bytes": [_vp],
    "tm_num_boxes": [_vp],
    "tm_path": [_vp],
    "tm_desc_size": [],
    "tm_pick_swizzle": [_u32],
}
for _name, _args in _SIGS.items():
    _f = getattr(_L, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_int
_L.tm_last_error.restype = ctypes.c_char_p
for _name in ("tm_box_bytes", "tm_num_boxes", "tm_desc_size"):
    getattr(_L, _name).restype = ctypes.c_size_t

if _L.tm_desc_size() != DESC_SIZE:
    raise ImportError("libtmap_gb300.so and its binding disagree on sizeof(tm_desc)")


class TmapError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = _L.tm_last_error().decode(errors="replace")
        super().__init__(f"{where} failed with status {code}: {msg}")
        self.code = code


def _check(rc: int, where: str) -> None:
    if rc != TM_OK:
        raise TmapError(rc, where)


def _addr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


class _Desc(ctypes.Structure):
    """Read-only mirror of the C tm_desc (field offsets are fixed by the ABI)."""
    _fields_ = [
        ("magic", _u32), ("dtype", _u32), ("esize", _u32), ("rank", _u32), ("swizzle", _u32),
        ("oob", _u32), ("path", _u32), ("why_fallback", _u32), ("base", _u64),
        ("dim", _u64 * 5), ("stride", _u64 * 5), ("box", _u32 * 5), ("estride", _u32 * 5),
        ("nbox", _u64 * 5), ("box_bytes", _u64), ("num_boxes", _u64),
        ("l2_promotion", ctypes.c_uint32), ("reserved", ctypes.c_uint8 * 36),
        ("tmap", ctypes.c_uint8 * 128),
    ]


assert ctypes.sizeof(_Desc) == DESC_SIZE


class TensorMap:
    """Owns a 64-byte aligned tm_desc (and keeps the described tensor alive)."""

    def __init__(self, keepalive=None):
        self._raw = ctypes.create_string_buffer(DESC_SIZE + 64)
        a = ctypes.addressof(self._raw)
        self.ptr = (a + 63) & ~63
        self.keepalive = keepalive

    @property
    def d(self) -> _Desc:
        return _Desc.from_address(self.ptr)

    @property
    def rank(self) -> int:
        return self.d.rank

    @property
    def box(self):
        return list(self.d.box[: self.rank])

    @property
    def dims(self):
        return list(self.d.dim[: self.rank])

    @property
    def box_bytes(self) -> int:
        return int(_L.tm_box_bytes(self.ptr))

    @property
    def num_boxes(self) -> int:
        return int(_L.tm_num_boxes(self.ptr))

    @property
    def path(self) -> int:
        return int(_L.tm_path(self.ptr))

    @property
    def base(self) -> int:
        """Device address of the tensor's element (0, ..., 0)."""
        return int(self.d.base)

    @property
    def why_fallback(self) -> int:
        return int(self.d.why_fallback)

    @property
    def l2_promotion(self) -> int:
        return int(self.d.l2_promotion)


def _arr(ctype, vals):
    vals = list(vals)
    return (ctype * max(len(vals), 1))(*vals)


def _make(fn, where, dtype, base, global_dim, global_strides, box_dim, element_strides, swizzle,
          oob) -> TensorMap:
    rank = len(global_dim)
    m = TensorMap(keepalive=None if isinstance(base, int) else base)
    es = None if element_strides is None else _arr(_u32, element_strides)
    rc = fn(m.ptr, int(dtype), rank, _addr(base), _arr(_u64, global_dim),
            _arr(_u64, global_strides or []), _arr(_u32, box_dim), es, int(swizzle), int(oob))
    _check(rc, where)
    return m


def tmap_plan(dtype, base, global_dim, global_strides, box_dim, element_strides=None,
              swizzle=TM_SWIZZLE_NONE, oob=TM_OOB_ZERO) -> TensorMap:
    return _make(_L.tmap_plan, "tmap_plan", dtype, base, global_dim, global_strides, box_dim,
                 element_strides, swizzle, oob)


def tmap_encode(dtype, base, global_dim, global_strides, box_dim, element_strides=None,
                swizzle=TM_SWIZZLE_NONE, oob=TM_OOB_ZERO) -> TensorMap:
    return _make(_L.tmap_encode, "tmap_encode", dtype, base, global_dim, global_strides, box_dim,
                 element_strides, swizzle, oob)


def tmap_replace_address(m: TensorMap, new_base) -> None:
    _check(_L.tmap_replace_address(m.ptr, _addr(new_base)), "tmap_replace_address")
    if not isinstance(new_base, int):
        m.keepalive = new_base


def tmap_force_fallback(m: TensorMap) -> None:
    _check(_L.tmap_force_fallback(m.ptr), "tmap_force_fallback")


def tmap_set_l2_promotion(m: TensorMap, promo: int) -> None:
    _check(_L.tmap_set_l2_promotion(m.ptr, int(promo)), "tmap_set_l2_promotion")


def _coords(coords, rank):
    flat = [int(v) for box in coords for v in box] if coords and isinstance(
        coords[0], (list, tuple)) else [int(v) for v in coords]
    if len(flat) % rank:
        raise ValueError("coordinate list length is not a multiple of the rank")
    return _arr(_i32, flat), len(flat) // rank


def tile_load_image(src: TensorMap, coords, image, stream=None) -> None:
    c, n = _coords(coords, src.rank)
    if n != 1:
        raise ValueError("tile_load_image takes one box")
    _check(_L.tile_load_image(src.ptr, c, _addr(image), _stream(stream)), "tile_load_image")


def tiled_copy(src: TensorMap, coords, images, stream=None) -> None:
    if coords is None:
        rc = _L.tiled_copy(src.ptr, None, 0, _addr(images), _stream(stream))
    else:
        c, n = _coords(coords, src.rank)
        rc = _L.tiled_copy(src.ptr, c, n, _addr(images), _stream(stream))
    _check(rc, "tiled_copy")


def tiled_copy_noalloc(src: TensorMap, coords, images, stream=None) -> None:
    """tiled_copy without any device allocation (fixed library-owned scratch; at most
    TM_NOALLOC_MAX_BOXES listed boxes); returns once the copy has finished."""
    if coords is None:
        rc = _L.tiled_copy_noalloc(src.ptr, None, 0, _addr(images), _stream(stream))
    else:
        c, n = _coords(coords, src.rank)
        rc = _L.tiled_copy_noalloc(src.ptr, c, n, _addr(images), _stream(stream))
    _check(rc, "tiled_copy_noalloc")


def tiled_roundtrip(dst: TensorMap, coords, images, stream=None) -> None:
    if coords is None:
        rc = _L.tiled_roundtrip(dst.ptr, None, 0, _addr(images), _stream(stream))
    else:
        c, n = _coords(coords, dst.rank)
        rc = _L.tiled_roundtrip(dst.ptr, c, n, _addr(images), _stream(stream))
    _check(rc, "tiled_roundtrip")


def tile_reduce_add(dst: TensorMap, src: TensorMap, stream=None) -> None:
    _check(_L.tile_reduce_add(dst.ptr, src.ptr, _stream(stream)), "tile_reduce_add")


def tile_reduce(dst: TensorMap, src: TensorMap, op, stream=None) -> None:
    _check(_L.tile_reduce(dst.ptr, src.ptr, int(op), _stream(stream)), "tile_reduce")


def stream_tiles(a: TensorMap, b: TensorMap, stages, cs_a, cs_b, bits_a, bits_b,
                 stream=None) -> None:
    _check(_L.stream_tiles(a.ptr, b.ptr, int(stages), _addr(cs_a), _addr(cs_b), _addr(bits_a),
                           _addr(bits_b), _stream(stream)), "stream_tiles")


def stream_gemm(a: TensorMap, b: TensorMap, c, ldc=None, stages: int = 7, stream=None) -> None:
    """C = A * B^T on the tensor cores: A map {K, M} box {64, 128}, B map {K, N} box {64, 256},
    c an fp32 device buffer of M rows, ldc elements apart (default N)."""
    ldc = b.dims[1] if ldc is None else ldc
    _check(_L.stream_gemm(a.ptr, b.ptr, _addr(c), int(ldc), int(stages), _stream(stream)),
           "stream_gemm")


def tm_stream_check(stream=None) -> int:
    """Returns the status code (TM_OK, TM_ETIMEOUT, ...) without raising."""
    return int(_L.tm_stream_check(_stream(stream)))


def tm_last_error() -> str:
    return _L.tm_last_error().decode(errors="replace")


def tm_selftest_wait_timeout(timeout_ns: int, stream=None) -> None:
    _check(_L.tm_selftest_wait_timeout(int(timeout_ns), _stream(stream)),
           "tm_selftest_wait_timeout")


def tm_pick_swizzle(inner_bytes: int) -> int:
    return int(_L.tm_pick_swizzle(int(inner_bytes)))
