"""CPU oracle for descriptor-driven tiled tensor movement (ctypes wrapper over tmap_oracle.c).

TEST INFRASTRUCTURE ONLY.  The oracle defines what the GPU path must compute and is written from
the pages' definitions; only the test suite, the smoke check and the benchmark's CPU-baseline leg
may import it.  It shares no code with the GPU library and never imports it.

Pin status per function is listed in tmap_oracle.h; the 64-byte and 32-byte swizzle layouts, which
the pages name without defining, are pinned by the chunk patterns NVIDIA's public CUDA
documentation gives for those modes.

All dimension lists here are innermost first.  A map views a numpy buffer: `buf` (any dtype, used
as raw bytes), a byte offset of element (0, ..., 0), dims, byte strides of dims 1..rank-1, the box
and a swizzle span (0, 32, 64 or 128).
"""
from __future__ import annotations

import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build

_LIB = None


class _OrcMap(ctypes.Structure):
    _fields_ = [
        ("esize", ctypes.c_uint32),
        ("rank", ctypes.c_uint32),
        ("span", ctypes.c_uint32),
        ("fill", ctypes.c_uint32),
        ("base", ctypes.c_void_p),
        ("dim", ctypes.c_uint64 * 5),
        ("stride", ctypes.c_int64 * 5),
        ("box", ctypes.c_uint32 * 5),
        ("estride", ctypes.c_uint32 * 5),
    ]


class _OrcMbar(ctypes.Structure):
    _fields_ = [
        ("count", ctypes.c_int64),
        ("pending", ctypes.c_int64),
        ("tx", ctypes.c_int64),
        ("phase", ctypes.c_uint32),
        ("completed", ctypes.c_uint32),
    ]


def lib():
    global _LIB
    if _LIB is None:
        # TMAP_ORACLE_LIB points the pins at a deliberately broken build (tests/test_oracle_mutants.py)
        path = os.environ.get("TMAP_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.POINTER
        u8p = ctypes.c_void_p
        L.orc_map_check.argtypes = [P(_OrcMap)]
        L.orc_swz.argtypes = [ctypes.c_uint64, ctypes.c_uint32]
        L.orc_swz.restype = ctypes.c_uint64
        L.orc_extent.argtypes = [P(_OrcMap), ctypes.c_uint32]
        L.orc_extent.restype = ctypes.c_uint32
        L.orc_box_bytes.argtypes = [P(_OrcMap)]
        L.orc_box_bytes.restype = ctypes.c_uint64
        L.orc_num_boxes.argtypes = [P(_OrcMap)]
        L.orc_num_boxes.restype = ctypes.c_uint64
        L.orc_box_start.argtypes = [P(_OrcMap), ctypes.c_uint64, P(ctypes.c_int32)]
        L.orc_image.argtypes = [P(_OrcMap), P(ctypes.c_int32), u8p]
        L.orc_store.argtypes = [P(_OrcMap), P(ctypes.c_int32), u8p]
        L.orc_reduce_add_f32.argtypes = [P(_OrcMap), P(ctypes.c_int32), u8p]
        L.orc_tiled_copy.argtypes = [P(_OrcMap), P(ctypes.c_int32), ctypes.c_uint64,
                                     ctypes.c_uint64, u8p]
        L.orc_tiled_roundtrip.argtypes = [P(_OrcMap), P(ctypes.c_int32), ctypes.c_uint64,
                                          ctypes.c_uint64, u8p]
        L.orc_tile_reduce_add.argtypes = [P(_OrcMap), P(_OrcMap), ctypes.c_uint64, ctypes.c_uint64]
        L.orc_combine.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int, ctypes.c_int]
        L.orc_combine.restype = ctypes.c_uint32
        L.orc_reduce_op.argtypes = [P(_OrcMap), P(ctypes.c_int32), u8p, ctypes.c_int, ctypes.c_int]
        L.orc_tile_reduce.argtypes = [P(_OrcMap), P(_OrcMap), ctypes.c_uint64, ctypes.c_uint64,
                                      ctypes.c_int, ctypes.c_int]
        L.orc_f16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_f16_to_double.restype = ctypes.c_double
        L.orc_f16_from_double.argtypes = [ctypes.c_double]
        L.orc_f16_from_double.restype = ctypes.c_uint16
        L.orc_bf16_from_double.argtypes = [ctypes.c_double]
        L.orc_bf16_from_double.restype = ctypes.c_uint16
        u64 = ctypes.c_uint64
        for name in ("orc_gemm_dot", "orc_gemm_dot_abs"):
            getattr(L, name).argtypes = [u8p, u64, u8p, u64, u64, u64, u64]
            getattr(L, name).restype = ctypes.c_double
        L.orc_gemm_block.argtypes = [u8p, u64, u8p, u64, u64, u64, u64, u64, u64, u8p]
        L.orc_tile_checksum.argtypes = [u8p, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                        P(ctypes.c_float), P(ctypes.c_uint64)]
        L.orc_stream_checksums.argtypes = [P(_OrcMap), P(_OrcMap), ctypes.c_uint64,
                                           ctypes.c_uint64, u8p, u8p, u8p, u8p]
        for name in ("orc_mbar_init", "orc_mbar_expect_tx", "orc_mbar_arrive_expect_tx",
                     "orc_mbar_complete_tx"):
            getattr(L, name).argtypes = [P(_OrcMbar), ctypes.c_uint32]
        L.orc_mbar_arrive.argtypes = [P(_OrcMbar)]
        L.orc_mbar_test_wait.argtypes = [P(_OrcMbar), ctypes.c_uint32]
        L.orc_bank_sectors.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int,
                                       P(ctypes.c_uint32)]
        _LIB = L
    return _LIB


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# out-of-bounds fill (values of the C enum): zero bytes, or the NaN of a float format
FILL_ZERO, FILL_NAN_F16, FILL_NAN_BF16, FILL_NAN_F32, FILL_NAN_F64 = 0, 1, 2, 3, 4


class Map:
    """A tensor map over a host numpy buffer, as the oracle sees it.  `estrides` are the
    elementStrides (default all 1); `fill` one of the FILL_* values."""

    def __init__(self, buf: np.ndarray, esize: int, dims, strides, box, span: int = 0,
                 offset: int = 0, estrides=None, fill: int = FILL_ZERO):
        rank = len(dims)
        estrides = [1] * rank if estrides is None else list(estrides)
        if not (1 <= rank <= 5) or len(box) != rank or len(strides) != rank - 1 \
                or len(estrides) != rank:
            raise ValueError("rank / dims / strides / box / estrides lengths disagree")
        if not buf.flags.c_contiguous:
            raise ValueError("buffer must be contiguous")
        self.buf = buf  # keep alive
        self.esize, self.dims, self.box, self.span = esize, list(dims), list(box), span
        self.estrides, self.fill = estrides, fill
        self.strides = [esize] + list(strides)
        s = _OrcMap()
        s.esize, s.rank, s.span, s.fill = esize, rank, span, fill
        s.base = _ptr(buf) + offset
        for i in range(5):
            s.dim[i] = dims[i] if i < rank else 1
            s.stride[i] = self.strides[i] if i < rank else 0
            s.box[i] = box[i] if i < rank else 1
            s.estride[i] = estrides[i] if i < rank else 1
        self.c = s
        rc = lib().orc_map_check(ctypes.byref(s))
        if rc != 0:
            raise ValueError(f"map not defined by the oracle (check code {rc})")

    @property
    def rank(self) -> int:
        return len(self.dims)

    def extent(self, i: int) -> int:
        """Image elements along dim i: ceil(box[i] / estride[i])."""
        return int(lib().orc_extent(ctypes.byref(self.c), i))

    @property
    def box_bytes(self) -> int:
        return int(lib().orc_box_bytes(ctypes.byref(self.c)))

    @property
    def num_boxes(self) -> int:
        return int(lib().orc_num_boxes(ctypes.byref(self.c)))

    def box_start(self, b: int):
        s = (ctypes.c_int32 * 5)()
        lib().orc_box_start(ctypes.byref(self.c), b, s)
        return [s[i] for i in range(self.rank)]


def _coords_arg(coords, rank):
    if coords is None:
        return None, None
    c = np.ascontiguousarray(np.asarray(coords, dtype=np.int32).reshape(-1, rank))
    return c, c.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def swz(off: int, span: int) -> int:
    return int(lib().orc_swz(off, span))


def image(m: Map, start) -> np.ndarray:
    s = (ctypes.c_int32 * 5)(*start)
    out = np.empty(m.box_bytes, dtype=np.uint8)
    lib().orc_image(ctypes.byref(m.c), s, _ptr(out))
    return out


def store(m: Map, start, img: np.ndarray) -> None:
    img = np.ascontiguousarray(img, dtype=np.uint8)
    s = (ctypes.c_int32 * 5)(*start)
    lib().orc_store(ctypes.byref(m.c), s, _ptr(img))


def _split(n: int, threads: int):
    threads = max(1, min(threads, n)) if n else 1
    step = (n + threads - 1) // threads if n else 0
    return [(i * step, min(n, (i + 1) * step)) for i in range(threads) if i * step < n]


def _run(fn, n: int, threads: int):
    """Run fn(b0, b1) over [0, n) split into contiguous ranges; ctypes releases the GIL, so the
    ranges run on separate cores."""
    ranges = _split(n, threads)
    if len(ranges) <= 1:
        for b0, b1 in ranges:
            fn(b0, b1)
        return
    with ThreadPoolExecutor(len(ranges)) as ex:
        list(ex.map(lambda r: fn(*r), ranges))


def tiled_copy(m: Map, coords=None, nbox: int | None = None, threads: int = 1,
               b0: int = 0, b1: int | None = None, out: np.ndarray | None = None) -> np.ndarray:
    c, cp = _coords_arg(coords, m.rank)
    n = m.num_boxes if c is None else c.shape[0]
    if nbox is not None:
        n = nbox
    b1 = n if b1 is None else b1
    if out is None:
        out = np.zeros(n * m.box_bytes, dtype=np.uint8)
    L = lib()
    _run(lambda x0, x1: L.orc_tiled_copy(ctypes.byref(m.c), cp, b0 + x0, b0 + x1, _ptr(out)),
         b1 - b0, threads)
    return out


def tiled_roundtrip(m: Map, images: np.ndarray, coords=None, threads: int = 1,
                    b0: int = 0, b1: int | None = None) -> None:
    c, cp = _coords_arg(coords, m.rank)
    n = m.num_boxes if c is None else c.shape[0]
    b1 = n if b1 is None else b1
    images = np.ascontiguousarray(images).view(np.uint8)
    L = lib()
    _run(lambda x0, x1: L.orc_tiled_roundtrip(ctypes.byref(m.c), cp, b0 + x0, b0 + x1,
                                              _ptr(images)), b1 - b0, threads)


def tile_reduce_add(dst: Map, src: Map, threads: int = 1, b0: int = 0,
                    b1: int | None = None) -> None:
    if dst.dims != src.dims or dst.box != src.box or dst.esize != 4 or src.esize != 4:
        raise ValueError("reduce-add needs fp32 maps with equal dims and box")
    b1 = dst.num_boxes if b1 is None else b1
    L = lib()
    _run(lambda x0, x1: L.orc_tile_reduce_add(ctypes.byref(dst.c), ctypes.byref(src.c),
                                              b0 + x0, b0 + x1), b1 - b0, threads)


# element types and operations of the general reduce (values of the C enums)
F32, F16, BF16, U32, S32 = 0, 1, 2, 3, 4
ADD, MIN, MAX = 0, 1, 2
TYPE_ESIZE = {F32: 4, F16: 2, BF16: 2, U32: 4, S32: 4}


def combine(a: int, b: int, type_: int, op: int) -> int:
    """Bit pattern of op(a, b) for one element (a from the destination, b from the source)."""
    return int(lib().orc_combine(a, b, type_, op))


def f16_from_double(v: float) -> int:
    return int(lib().orc_f16_from_double(v))


def bf16_from_double(v: float) -> int:
    return int(lib().orc_bf16_from_double(v))


def f16_to_double(h: int) -> float:
    return float(lib().orc_f16_to_double(h))


def tile_reduce(dst: Map, src: Map, type_: int, op: int, threads: int = 1, b0: int = 0,
                b1: int | None = None) -> None:
    """dst = op(dst, src) over boxes b0..b1-1 of dst's grid (src: same dims and box)."""
    if dst.dims != src.dims or dst.box != src.box:
        raise ValueError("reduce needs maps with equal dims and box")
    if dst.esize != TYPE_ESIZE[type_] or src.esize != TYPE_ESIZE[type_]:
        raise ValueError("element size does not match the reduce type")
    b1 = dst.num_boxes if b1 is None else b1
    L = lib()
    _run(lambda x0, x1: L.orc_tile_reduce(ctypes.byref(dst.c), ctypes.byref(src.c), b0 + x0,
                                          b0 + x1, type_, op), b1 - b0, threads)


def _bf16_matrix(x: np.ndarray, name: str) -> np.ndarray:
    if x.dtype != np.uint16 or x.ndim != 2 or not x.flags.c_contiguous:
        raise ValueError(f"{name} must be a C-contiguous 2-D uint16 (bf16 bits) array")
    return x


def gemm(a: np.ndarray, b: np.ndarray, m0: int = 0, m1: int | None = None, n0: int = 0,
         n1: int | None = None, k: int | None = None) -> np.ndarray:
    """C[m][n] = sum_k A[m][k] * B[n][k] in double, for bf16 bit arrays A (M x K) and B (N x K);
    the block [m0, m1) x [n0, n1)."""
    a, b = _bf16_matrix(a, "a"), _bf16_matrix(b, "b")
    k = a.shape[1] if k is None else k
    if k > a.shape[1] or k > b.shape[1]:
        raise ValueError("k exceeds a row")
    m1 = a.shape[0] if m1 is None else m1
    n1 = b.shape[0] if n1 is None else n1
    out = np.zeros((m1 - m0, n1 - n0), np.float64)
    lib().orc_gemm_block(_ptr(a), a.shape[1], _ptr(b), b.shape[1], k, m0, m1, n0, n1, _ptr(out))
    return out


def gemm_entry(a: np.ndarray, b: np.ndarray, m: int, n: int):
    """(C[m][n], sum_k |A[m][k] * B[n][k]|), both in double."""
    a, b = _bf16_matrix(a, "a"), _bf16_matrix(b, "b")
    L = lib()
    args = (_ptr(a), a.shape[1], _ptr(b), b.shape[1], a.shape[1], m, n)
    return float(L.orc_gemm_dot(*args)), float(L.orc_gemm_dot_abs(*args))


def tile_checksum(img: np.ndarray, rows: int, row_bytes: int, span: int):
    img = np.ascontiguousarray(img, dtype=np.uint8)
    cs = ctypes.c_float()
    bits = ctypes.c_uint64()
    lib().orc_tile_checksum(_ptr(img), rows, row_bytes, span, ctypes.byref(cs), ctypes.byref(bits))
    return np.float32(cs.value), int(bits.value)


def stream_checksums(a: Map, b: Map, threads: int = 1, t0: int = 0, t1: int | None = None):
    if a.num_boxes != b.num_boxes:
        raise ValueError("A and B must have the same number of tiles")
    n = a.num_boxes
    t1 = n if t1 is None else t1
    cs_a = np.zeros(n, np.float32)
    cs_b = np.zeros(n, np.float32)
    bits_a = np.zeros(n, np.uint64)
    bits_b = np.zeros(n, np.uint64)
    L = lib()
    _run(lambda x0, x1: L.orc_stream_checksums(ctypes.byref(a.c), ctypes.byref(b.c), t0 + x0,
                                               t0 + x1, _ptr(cs_a), _ptr(cs_b), _ptr(bits_a),
                                               _ptr(bits_b)), t1 - t0, threads)
    return cs_a, cs_b, bits_a, bits_b


class Mbar:
    """mbarrier phase model (arrival count, pending transaction bytes, phase parity)."""

    def __init__(self, count: int):
        self.c = _OrcMbar()
        lib().orc_mbar_init(ctypes.byref(self.c), count)

    def expect_tx(self, n):
        lib().orc_mbar_expect_tx(ctypes.byref(self.c), n)

    def arrive(self):
        lib().orc_mbar_arrive(ctypes.byref(self.c))

    def arrive_expect_tx(self, n):
        lib().orc_mbar_arrive_expect_tx(ctypes.byref(self.c), n)

    def complete_tx(self, n):
        lib().orc_mbar_complete_tx(ctypes.byref(self.c), n)

    def test_wait(self, parity) -> bool:
        return bool(lib().orc_mbar_test_wait(ctypes.byref(self.c), parity))

    @property
    def pending(self):
        return self.c.pending

    @property
    def tx(self):
        return self.c.tx

    @property
    def phase(self):
        return self.c.phase


def bank_sectors(col: int, row0: int, grouped: bool):
    out = (ctypes.c_uint32 * 8)()
    lib().orc_bank_sectors(col, row0, 1 if grouped else 0, out)
    return [out[i] for i in range(8)]


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
