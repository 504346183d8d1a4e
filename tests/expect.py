"""Expected values built from library routines and the pages' printed rules, independent of the
oracle's own arithmetic.  Used to pin the oracle (and nothing here is used by the GPU path).

- `strided_view`: numpy's as_strided over a byte buffer: the textbook meaning of dims + strides.
- `box_none`: the box of a zero-padded tensor, taken with numpy fancy indexing.
- `apply_page_swizzle128`: the rule of mlc.ai "Modern GPU Programming for MLSys", chapter
  "异步数据搬运：TMA", §"用 3D TMA 搬运多个 swizzle atoms": in each 8-row x 128-byte atom, logical
  sector c of row r goes to physical sector c XOR (r % 8).  Applied through a table read from the
  golden fixture, not through address bits.
"""
from __future__ import annotations

import os

import numpy as np

_ROOT = os.path.dirname(os.path.abspath(__file__))

_NP_UINT = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}


def sector_table():
    rows = []
    with open(os.path.join(_ROOT, "golden", "mlsys_swizzle128_sector_table.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                rows.append([int(v) for v in ln.split()])
    t = np.array(rows, dtype=np.int64)
    assert t.shape == (8, 8)
    return t


def strided_view(buf: np.ndarray, offset: int, esize: int, dims, strides_bytes) -> np.ndarray:
    """numpy view of the global tensor: shape outermost first, byte strides from the map."""
    raw = buf.reshape(-1).view(np.uint8)
    dt = _NP_UINT[esize]
    shape = tuple(reversed(dims))
    strides = tuple(reversed([esize] + list(strides_bytes)))
    return np.lib.stride_tricks.as_strided(raw[offset:].view(dt), shape=shape, strides=strides,
                                           writeable=False)


def box_none(view: np.ndarray, start, box) -> np.ndarray:
    """Elements of the box (innermost-first start/box) with zeros outside the tensor; returned
    outermost first, i.e. in image order."""
    rank = len(box)
    dims = list(reversed(view.shape))
    idx, ok = [], []
    for i in reversed(range(rank)):
        g = start[i] + np.arange(box[i])
        ok.append((g >= 0) & (g < dims[i]))
        idx.append(np.clip(g, 0, max(dims[i] - 1, 0)))
    vals = view[np.ix_(*idx)].copy()
    mask = np.ones(vals.shape, dtype=bool)
    for ax, o in enumerate(ok):
        shp = [1] * rank
        shp[ax] = len(o)
        mask &= o.reshape(shp)
    vals[~mask] = 0
    return vals


def inbounds_mask(dims, start, box) -> np.ndarray:
    rank = len(box)
    mask = np.ones(tuple(reversed(box)), dtype=bool)
    for ax, i in enumerate(reversed(range(rank))):
        g = start[i] + np.arange(box[i])
        shp = [1] * rank
        shp[ax] = box[i]
        mask &= ((g >= 0) & (g < dims[i])).reshape(shp)
    return mask


def apply_page_swizzle128(none_bytes: np.ndarray) -> np.ndarray:
    """Place the sectors of an unswizzled image of 128-byte rows per the page's rule."""
    t = sector_table()
    rows = none_bytes.reshape(-1, 8, 16)
    out = np.empty_like(rows)
    for r in range(rows.shape[0]):
        for c in range(8):
            out[r, t[r % 8, c]] = rows[r, c]
    return out.reshape(-1)


def checksum_reference(logical_rows: np.ndarray):
    """fp32 checksum of a bf16 tile given as logical rows of uint16 bit patterns: sequential row
    sums via numpy's accumulate (one rounding per step, in order), then a pairwise tree."""
    f = (logical_rows.astype(np.uint32) << np.uint32(16)).view(np.float32)
    sums = np.add.accumulate(f, axis=1, dtype=np.float32)[:, -1].copy()
    while sums.size > 1:
        sums = (sums[0::2] + sums[1::2]).astype(np.float32)
    bits = int(logical_rows.astype(np.uint64).sum())
    return np.float32(sums[0]), bits


def box_stepped(view: np.ndarray, start, box, estrides, fill=0):
    """Image elements of a box with element strides, outermost first: along dim i the elements
    start[i], start[i] + estrides[i], ... below start[i] + box[i], taken with numpy basic slicing
    (step estrides[i]) of the tensor padded by `fill` on every side; also returns the in-bounds
    mask of the same shape."""
    rank = len(box)
    pad = [(max(box[i], 1) + abs(start[i]), max(box[i], 1) + abs(start[i]))
           for i in reversed(range(rank))]
    padded = np.pad(np.ascontiguousarray(view), pad, constant_values=fill)
    inside = np.pad(np.ones(view.shape, dtype=bool), pad, constant_values=False)
    sl = tuple(slice(start[i] + pad[rank - 1 - i][0], start[i] + pad[rank - 1 - i][0] + box[i],
                     estrides[i]) for i in reversed(range(rank)))
    return padded[sl].copy(), inside[sl].copy()
