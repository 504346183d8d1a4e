"""Seeded synthetic inputs for descriptor-driven tiled tensor movement.

This module only makes input bytes and describes the workloads' shapes; it holds none of the
method's arithmetic (no swizzle, no box addressing, no reduction).  Both the CPU oracle's tests
and the GPU path's tests and benchmark draw their inputs from here, so that both sides see the same
bytes.

Shapes follow the pages' examples ([MLSys-TMA] = mlc.ai "Modern GPU Programming for MLSys",
chapter "异步数据搬运：TMA"):
  W1  fp16 16 x 128, element (r, c) holds the bit pattern r*128 + c; one 8 x 64 box at (0, 0) and
      at column 64 / row 8 (§"异步数据搬运：TMA", the interactive figure's 16 x 128 tensor and 8 x 64
      tile).
  W2  fp16 16 x 256 viewed as (group, row, col) slices of 128 columns (§"用 3D TMA 搬运多个 swizzle
      atoms"), seeded random bit patterns that are never NaN or Inf.
  W3  bf16 8192 x 8192, normal(0, 1) rounded to bf16, 128 x 64 boxes, 128-byte swizzle.
  W4  bf16 16 x 4095 x 1000 stored with a padded row of 1024 elements (2048 bytes); the padding
      holds the sentinel 0xDEAD.  Ragged 64 x 64 / 64 x 32 boxes and a rank-5 view
      4 x 4 x 4095 x 10 x 100 whose 200-byte stride no tensor-map hardware can take.
  W5a fp32 16384 x 16384 destination normal(0, 1) and source uniform(-1, 1), 128 x 32 boxes.
  W5b bf16 A 8192 x 4096 and B 4096 x 8192, 128 x 64 tiles streamed through a 4-stage ring.

Every shape list in this module is outermost first (how a user writes a matrix); the maps built
from them list dims innermost first, as the tensor-map encoder wants.
"""
from __future__ import annotations

import numpy as np

SENTINEL_U16 = 0xDEAD

SEEDS = {"w2": 2, "w3": 3, "w4": 4, "w5a_dst": 51, "w5a_src": 52, "w5b_a": 53, "w5b_b": 54}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); returns uint16 bits.
    Inputs are finite by construction."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def normal_bf16(shape, seed: int) -> np.ndarray:
    """bf16 bit patterns of normal(0, 1) draws, shape outermost first."""
    rng = np.random.default_rng(seed)
    out = np.empty(int(np.prod(shape)), dtype=np.uint16)
    chunk = 1 << 22
    for i in range(0, out.size, chunk):
        n = min(chunk, out.size - i)
        out[i:i + n] = f32_to_bf16_bits(rng.standard_normal(n, dtype=np.float32))
    return out.reshape(shape)


def finite_f16_bits(shape, seed: int) -> np.ndarray:
    """Uniform 16-bit patterns, redrawn wherever the fp16 exponent field is all ones (NaN / Inf)."""
    rng = np.random.default_rng(seed)
    x = rng.integers(0, 1 << 16, size=shape, dtype=np.uint32).astype(np.uint16)
    while True:
        bad = (x & 0x7C00) == 0x7C00
        if not bad.any():
            return x
        x[bad] = rng.integers(0, 1 << 16, size=int(bad.sum()), dtype=np.uint32).astype(np.uint16)


def w1_tensor() -> np.ndarray:
    """fp16 16 x 128 whose element (r, c) carries the bit pattern r*128 + c."""
    r = np.arange(16, dtype=np.uint32)[:, None]
    c = np.arange(128, dtype=np.uint32)[None, :]
    return (r * 128 + c).astype(np.uint16)


def w2_tensor(seed: int = SEEDS["w2"]) -> np.ndarray:
    return finite_f16_bits((16, 256), seed)


def w3_tensor(rows: int = 8192, cols: int = 8192, seed: int = SEEDS["w3"]) -> np.ndarray:
    return normal_bf16((rows, cols), seed)


def w4_tensor(batch: int = 16, rows: int = 4095, cols: int = 1000, pitch: int = 1024,
              seed: int = SEEDS["w4"]) -> np.ndarray:
    """bf16 batch x rows x cols stored with a row pitch of `pitch` elements; the padding columns
    cols..pitch-1 hold the sentinel."""
    x = np.full((batch, rows, pitch), SENTINEL_U16, dtype=np.uint16)
    x[:, :, :cols] = normal_bf16((batch, rows, cols), seed)
    return x


TINY_F32 = np.float32(2.0 ** -126)  # smallest normal binary32


def w5a_tensors(rows: int = 16384, cols: int = 16384, seed_dst: int = SEEDS["w5a_dst"],
                seed_src: int = SEEDS["w5a_src"]):
    """fp32 destination normal(0, 1) and source uniform(-1, 1) (2u - 1 with u uniform on [0, 1),
    exact in float32).  Pairs whose operands or exact sum would be subnormal are redrawn, so
    flush-to-zero can never decide a result."""
    rd = np.random.default_rng(seed_dst)
    rs = np.random.default_rng(seed_src)
    dst = np.empty((rows, cols), dtype=np.float32)
    src = np.empty((rows, cols), dtype=np.float32)
    fd = dst.reshape(-1)
    fs = src.reshape(-1)
    chunk = 1 << 22
    for i in range(0, fd.size, chunk):
        d = fd[i:i + chunk]
        s = fs[i:i + chunk]
        rd.standard_normal(d.size, dtype=np.float32, out=d)
        rs.random(s.size, dtype=np.float32, out=s)
        s *= 2
        s -= 1
        while True:
            # Both operands are multiples of 2^-149, so a sum below 2^-126 in magnitude is exactly
            # representable and the float32 sum equals the exact one there.
            tot = d + s
            bad = (((np.abs(d) < TINY_F32) & (d != 0)) | ((np.abs(s) < TINY_F32) & (s != 0))
                   | ((np.abs(tot) < TINY_F32) & (tot != 0)))
            if not bad.any():
                break
            nb = int(bad.sum())
            s[bad] = rs.random(nb, dtype=np.float32) * np.float32(2) - np.float32(1)
            d[bad] = rd.standard_normal(nb, dtype=np.float32)
    return dst, src


def w5b_tensors(m: int = 8192, k: int = 4096, n: int = 8192, seed_a: int = SEEDS["w5b_a"],
                seed_b: int = SEEDS["w5b_b"]):
    """bf16 A (m x k) and B (k x n)."""
    return normal_bf16((m, k), seed_a), normal_bf16((k, n), seed_b)


def reduce_operands(kind: str, rows: int, cols: int, seed: int):
    """Destination and source bit patterns (rows x cols) for the general reduce, kind one of
    f32, f16, bf16 (normal(0, 1) values, then no zeros and no pair whose exact sum is a nonzero
    subnormal), u32, s32 (uniform 32-bit patterns)."""
    rng = np.random.default_rng(seed)
    if kind in ("u32", "s32"):
        d = rng.integers(0, 1 << 32, size=(rows, cols), dtype=np.uint64).astype(np.uint32)
        s = rng.integers(0, 1 << 32, size=(rows, cols), dtype=np.uint64).astype(np.uint32)
        return (d, s) if kind == "u32" else (d.view(np.int32), s.view(np.int32))

    def draw(n):
        v = rng.standard_normal(n).astype(np.float32)
        if kind == "f32":
            return v.view(np.uint32)
        if kind == "f16":
            return v.astype(np.float16).view(np.uint16)
        return f32_to_bf16_bits(v)

    def value(bits):
        if kind == "f32":
            return bits.view(np.float32).astype(np.float64)
        if kind == "f16":
            return bits.view(np.float16).astype(np.float64)
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)

    tiny = {"f32": 2.0 ** -126, "f16": 2.0 ** -14, "bf16": 2.0 ** -126}[kind]
    d, s = draw(rows * cols), draw(rows * cols)
    while True:
        vd, vs = value(d), value(s)
        tot = vd + vs
        bad = (vd == 0) | (vs == 0) | ((np.abs(tot) < tiny) & (tot != 0))
        if not bad.any():
            return d.reshape(rows, cols), s.reshape(rows, cols)
        n = int(bad.sum())
        d[bad], s[bad] = draw(n), draw(n)


# Bit patterns of the special values of each float format: zeros, the smallest and largest
# subnormals, the smallest normal, one, the largest finite, infinities and quiet NaNs, both signs.
SPECIAL_BITS = {
    "f32": [0x00000000, 0x80000000, 0x00000001, 0x80000001, 0x007FFFFF, 0x807FFFFF, 0x00800000,
            0x80800000, 0x3F800000, 0xBF800000, 0x7F7FFFFF, 0xFF7FFFFF, 0x7F800000, 0xFF800000,
            0x7FC00000, 0xFFC00001],
    "f16": [0x0000, 0x8000, 0x0001, 0x8001, 0x03FF, 0x83FF, 0x0400, 0x8400, 0x3C00, 0xBC00,
            0x7BFF, 0xFBFF, 0x7C00, 0xFC00, 0x7E00, 0xFE01],
    "bf16": [0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x807F, 0x0080, 0x8080, 0x3F80, 0xBF80,
             0x7F7F, 0xFF7F, 0x7F80, 0xFF80, 0x7FC0, 0xFFC1],
    "u32": [0, 1, 2, 0x7FFFFFFF, 0x80000000, 0x80000001, 0xFFFFFFFE, 0xFFFFFFFF],
    "s32": [0, 1, 2, 0x7FFFFFFF, 0x80000000, 0x80000001, 0xFFFFFFFE, 0xFFFFFFFF],
}


def special_reduce_operands(kind: str, rows: int, cols: int, seed: int):
    """Destination and source bit patterns (rows x cols) for the general reduce at the formats'
    edges: the first len(SPECIAL_BITS[kind])^2 elements hold every (dst, src) pair of special
    patterns, the rest a seeded mix of special patterns, their neighbours (one unit in the last
    place up) and uniform random patterns."""
    rng = np.random.default_rng(seed)
    sp = np.array(SPECIAL_BITS[kind], dtype=np.uint64)
    width = 32 if kind in ("f32", "u32", "s32") else 16
    n = rows * cols
    pick = rng.integers(0, 3, size=(2, n))
    cand = np.stack([sp[rng.integers(0, len(sp), size=(2, n))],
                     (sp[rng.integers(0, len(sp), size=(2, n))] + 1) % (1 << width),
                     rng.integers(0, 1 << width, size=(2, n), dtype=np.uint64)])
    v = np.take_along_axis(cand, pick[None], axis=0)[0]
    k = len(sp)
    v[0, :k * k] = np.repeat(sp, k)[:n]
    v[1, :k * k] = np.tile(sp, k)[:n]
    dt = np.uint32 if width == 32 else np.uint16
    d, s = v[0].astype(dt).reshape(rows, cols), v[1].astype(dt).reshape(rows, cols)
    return (d.view(np.int32), s.view(np.int32)) if kind == "s32" else (d, s)


# Map recipes, dims innermost first: (dims, byte strides of dims 1.., box, swizzle span)
def w3_map(rows: int = 8192, cols: int = 8192, span: int = 128):
    return dict(dims=[cols, rows], strides=[cols * 2], box=[64, 128], span=span, esize=2)


def w4_rank3_map(box_cols: int, batch=16, rows=4095, cols=1000, pitch=1024, span=128):
    return dict(dims=[cols, rows, batch], strides=[pitch * 2, rows * pitch * 2],
                box=[box_cols, 64, 1], span=span, esize=2)


def w4_rank5_map(batch=16, rows=4095, cols=1000, pitch=1024, span=0):
    """The 4 x 4 x rows x 10 x 100 view: batch split 4 x 4, each row's first 1000 columns split
    into 10 groups of 100 (a 200-byte group stride)."""
    assert batch == 16 and cols == 1000
    return dict(dims=[100, 10, rows, 4, 4],
                strides=[200, pitch * 2, rows * pitch * 2, 4 * rows * pitch * 2],
                box=[64, 10, 32, 1, 1], span=span, esize=2)


def w5a_map(rows=16384, cols=16384, span=128):
    return dict(dims=[cols, rows], strides=[cols * 4], box=[32, 128], span=span, esize=4)


def w5b_maps(m=8192, k=4096, n=8192, span=128):
    a = dict(dims=[k, m], strides=[k * 2], box=[64, 128], span=span, esize=2)
    b = dict(dims=[n, k], strides=[n * 2], box=[64, 128], span=span, esize=2)
    return a, b


# Descriptor features over the W3 tensor (8192 x 8192 bf16): elementStrides take every other row
# (box 64 x 128, steps {1, 2}: 64 x 64 images, 128B swizzle) or every other column (box 128 x 64,
# steps {2, 1}: 64 x 64 images, no swizzle -- a swizzled map needs a unit innermost step).
def w6_rows2_map(rows: int = 8192, cols: int = 8192):
    return dict(w3_map(rows, cols, 128), estrides=[1, 2])


def w6_cols2_map(rows: int = 8192, cols: int = 8192):
    return dict(w3_map(rows, cols, 0), box=[128, 64], estrides=[2, 1])


# The ring in GEMM order (stream_gemm): A 8192 x 4096 and B 8192 x 4096 (B holds B^T: N x K, K
# contiguous), normal(0,1) rounded to bf16; C = A * B^T is 8192 x 8192 fp32.
SEEDS_W7 = (71, 72)


def w7_operands(m: int = 8192, n: int = 8192, k: int = 4096):
    return normal_bf16((m, k), SEEDS_W7[0]), normal_bf16((n, k), SEEDS_W7[1])
