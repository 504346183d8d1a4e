"""Helpers for the GPU parity tests: one map recipe, built on both sides (the C-ABI library over a
device buffer, the oracle over the same bytes on the host)."""
from __future__ import annotations

import numpy as np

import oracle

SPAN_TO_SW = {0: 0, 32: 1, 64: 2, 128: 3}
ESIZE_TO_DTYPE = {1: 0, 2: 9, 4: 7, 8: 4}  # u8, bf16, f32, u64: copies are bitwise


# Canary guard bands: every device buffer a test hands to the library (inputs, images, sentinel
# destinations) sits between two GUARD-byte bands of CANARY bytes; check_guards() (run after every
# test by the autouse fixture in conftest.py) fails the test if a kernel wrote into one.
GUARD = 4096
CANARY = 0xE7
_guarded = []


def guarded(nbytes: int, fill: int):
    """A uint8 device tensor of nbytes (16-byte aligned: the bands are 4 KiB) filled with `fill`,
    inside a larger buffer whose GUARD bytes on each side hold CANARY."""
    import torch
    buf = torch.full((GUARD + nbytes + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
    body = buf[GUARD:GUARD + nbytes]
    body.fill_(fill)
    _guarded.append((buf, nbytes))
    return body


def check_guards():
    """Every guard band still holds its canary bytes; forgets the buffers afterwards."""
    import torch
    try:
        for buf, nbytes in _guarded:
            lo, hi = buf[:GUARD], buf[GUARD + nbytes:]
            assert bool((lo == CANARY).all()) and bool((hi == CANARY).all()), (
                f"a kernel wrote into the guard band of a {nbytes}-byte buffer")
    finally:
        _guarded.clear()
        torch.cuda.synchronize()


def to_dev(arr: np.ndarray):
    import torch
    flat = np.ascontiguousarray(arr).reshape(-1).view(np.uint8)
    t = guarded(flat.size, 0)
    t.copy_(torch.from_numpy(flat))
    return t


def full_like(t, fill: int):
    """A guarded device buffer of t's byte size filled with `fill` (a sentinel destination)."""
    return guarded(t.numel() * t.element_size(), fill)


def to_host(t) -> np.ndarray:
    return t.cpu().numpy()


# library dtype code (TM_F16, TM_F32, TM_F64, TM_BF16) -> the oracle's NaN fill of that format
DTYPE_TO_NAN_FILL = {6: oracle.FILL_NAN_F16, 7: oracle.FILL_NAN_F32, 8: oracle.FILL_NAN_F64,
                     9: oracle.FILL_NAN_BF16}


def dev_map(tm, buf, r, offset=0, dtype=None):
    """Recipe keys: dims, strides, box, span, esize; optional estrides and nan (True: NaN fill)."""
    dt = ESIZE_TO_DTYPE[r["esize"]] if dtype is None else dtype
    m = tm.tmap_encode(dt, buf.data_ptr() + offset, r["dims"], r["strides"], r["box"],
                       element_strides=r.get("estrides"), swizzle=SPAN_TO_SW[r["span"]],
                       oob=tm.TM_OOB_NAN if r.get("nan") else tm.TM_OOB_ZERO)
    m.keepalive = buf  # the map holds a raw address: keep the tensor it points into alive
    return m


def host_map(arr: np.ndarray, r, offset=0, dtype=None):
    fill = DTYPE_TO_NAN_FILL[dtype] if r.get("nan") else oracle.FILL_ZERO
    return oracle.Map(arr, r["esize"], r["dims"], r["strides"], r["box"], r["span"],
                      offset=offset, estrides=r.get("estrides"), fill=fill)


def empty_images(n_boxes: int, box_bytes: int, fill: int = 0x5A):
    return guarded(n_boxes * box_bytes, fill)


U = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}
ESIZE = {6: 2, 9: 2, 7: 4, 8: 8}  # library dtype code -> element size


def as_float(bits, dtype, tm):
    if dtype == tm.TM_BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32)
    return bits.view({tm.TM_F16: np.float16, tm.TM_F32: np.float32, tm.TM_F64: np.float64}[dtype])


def assert_nan_fill(got, want, dtype, tm):
    """In-bounds elements (finite in the oracle's image) bit-exact; the rest NaN (the pages name
    no NaN bit pattern: any NaN is a correct fill)."""
    es = ESIZE[dtype]
    g, w = got.view(U[es]), want.view(U[es])
    oob = np.isnan(as_float(w, dtype, tm))
    assert oob.any() and (~oob).any()
    np.testing.assert_array_equal(g[~oob], w[~oob])
    assert np.isnan(as_float(g[oob], dtype, tm)).all()
