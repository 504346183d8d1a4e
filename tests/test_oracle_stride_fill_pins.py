"""Pins of two descriptor features of the oracle, no GPU needed:

- elementStrides -- fangpin "gpu-hpc-book", ch. 08 "Cuda TMA", §"Tensor descriptor：CUtensorMap":
  the step between the elements taken along each dim when the box is written to shared memory,
  counted in elements, not bytes.  Read here as: along dim i the image keeps the box's elements
  start, start + es, start + 2 es, ... below start + box, i.e. ceil(box / es) of them, packed.
  Pinned against numpy basic slicing with a step of the zero-padded tensor.
- out-of-bounds NaN fill -- coolgpu "H200 · TMA · Tensor Memory Accelerator", §02 (out-of-bounds
  elements are filled by the hardware with 0 or NaN).  Any NaN is accepted at those positions.
"""
import numpy as np
import pytest

import oracle
from expect import apply_page_swizzle128, box_stepped, strided_view

NP_UINT = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}


def rand_tensor(rng, esize, dims, pad_elems):
    """A tensor with padded rows: dim-0 pitch dims[0] + pad elements, dims outer packed."""
    pitch = dims[0] + pad_elems
    outer = int(np.prod(dims[1:])) if len(dims) > 1 else 1
    buf = rng.integers(1, 1 << min(8 * esize, 62), size=pitch * outer,
                       dtype=np.uint64).astype(NP_UINT[esize])
    strides, acc = [], pitch * esize
    for d in dims[1:]:
        strides.append(acc)
        acc *= d
    return buf, strides


def random_case(rng):
    rank = int(rng.integers(1, 5))
    esize = int(rng.choice([1, 2, 4, 8]))
    dims = [int(rng.integers(1, 30)) for _ in range(rank)]
    box = [int(rng.integers(1, 20)) for _ in range(rank)]
    es = [int(rng.integers(1, 9)) for _ in range(rank)]
    start = [int(rng.integers(-box[i], dims[i])) for i in range(rank)]
    return esize, dims, box, es, start


@pytest.mark.parametrize("seed", range(40))
def test_strided_image_is_numpy_step_slice(seed):
    rng = np.random.default_rng(100 + seed)
    esize, dims, box, es, start = random_case(rng)
    buf, strides = rand_tensor(rng, esize, dims, int(rng.integers(0, 5)))
    m = oracle.Map(buf, esize, dims, strides, box, estrides=es)
    want, _ = box_stepped(strided_view(buf, 0, esize, dims, strides), start, box, es)
    assert m.box_bytes == want.size * esize
    for i in range(len(dims)):
        assert m.extent(i) == -(-box[i] // es[i])
    got = oracle.image(m, start).view(NP_UINT[esize])
    np.testing.assert_array_equal(got, want.reshape(-1))


def test_units_are_elements_not_bytes():
    """f32 0, 1, 2, ...: a step of 2 takes elements 0, 2, 4, ... (8 bytes apart)."""
    x = np.arange(64, dtype=np.float32)
    m = oracle.Map(x, 4, [64], [], [16], estrides=[2])
    np.testing.assert_array_equal(oracle.image(m, [0]).view(np.float32),
                                  np.arange(0, 16, 2, dtype=np.float32))
    m3 = oracle.Map(x, 4, [64], [], [10], estrides=[3])  # ceil(10 / 3) = 4 elements
    np.testing.assert_array_equal(oracle.image(m3, [60]).view(np.float32),
                                  np.array([60, 63, 0, 0], dtype=np.float32))


def test_outer_step_skips_rows():
    x = np.arange(12 * 8, dtype=np.uint16).reshape(12, 8)
    m = oracle.Map(x, 2, [8, 12], [16], [8, 6], estrides=[1, 3])
    got = oracle.image(m, [0, 6]).view(np.uint16).reshape(2, 8)
    np.testing.assert_array_equal(got, x[[6, 9]])


def test_grid_is_independent_of_steps():
    buf = np.zeros(100 * 40, np.uint32)
    a = oracle.Map(buf, 4, [100, 40], [400], [8, 6])
    b = oracle.Map(buf, 4, [100, 40], [400], [8, 6], estrides=[4, 5])
    assert a.num_boxes == b.num_boxes == 13 * 7
    assert [b.box_start(k) for k in (0, 14, 90)] == [a.box_start(k) for k in (0, 14, 90)]
    assert b.box_bytes == 4 * 2 * 2


@pytest.mark.parametrize("seed", range(20))
def test_strided_store_writes_exactly_the_taken_positions(seed):
    rng = np.random.default_rng(300 + seed)
    esize, dims, box, es, start = random_case(rng)
    buf, strides = rand_tensor(rng, esize, dims, int(rng.integers(0, 4)))
    m = oracle.Map(buf, esize, dims, strides, box, estrides=es)
    img = rng.integers(0, 256, m.box_bytes, dtype=np.uint64).astype(np.uint8)
    dst = np.full_like(buf, 0x5A if esize == 1 else 0x5A5A)
    md = oracle.Map(dst, esize, dims, strides, box, estrides=es)
    oracle.store(md, start, img)
    # expected: a numbered tensor tells which position each image element maps to
    idx = np.arange(buf.size, dtype=np.int64)
    pos, ok = box_stepped(strided_view(idx.view(np.uint64), 0, 8, dims,
                                       [s // esize * 8 for s in strides]), start, box, es)
    want = np.full_like(buf, 0x5A if esize == 1 else 0x5A5A)
    vals = img.view(NP_UINT[esize]).reshape(pos.shape)
    want[pos[ok].astype(np.int64)] = vals[ok]
    np.testing.assert_array_equal(dst, want)


def test_strided_outer_dims_under_128b_swizzle():
    rng = np.random.default_rng(7)
    dims, box, es = [64, 40, 5], [64, 16, 3], [1, 3, 2]
    buf, strides = rand_tensor(rng, 2, dims, 8)
    for start in ([0, 0, 0], [0, 32, 3], [0, -6, -1]):
        none = oracle.image(oracle.Map(buf, 2, dims, strides, box, estrides=es), start)
        sw = oracle.image(oracle.Map(buf, 2, dims, strides, box, span=128, estrides=es), start)
        np.testing.assert_array_equal(sw, apply_page_swizzle128(none))
        want, _ = box_stepped(strided_view(buf, 0, 2, dims, strides), start, box, es)
        np.testing.assert_array_equal(none.view(np.uint16), want.reshape(-1))


def as_float(bits: np.ndarray, fill):
    if fill == oracle.FILL_NAN_BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32)
    return bits.view({oracle.FILL_NAN_F16: np.float16, oracle.FILL_NAN_F32: np.float32,
                      oracle.FILL_NAN_F64: np.float64}[fill])


@pytest.mark.parametrize("fill,esize", [(oracle.FILL_NAN_F16, 2), (oracle.FILL_NAN_BF16, 2),
                                        (oracle.FILL_NAN_F32, 4), (oracle.FILL_NAN_F64, 8)])
def test_nan_fill_marks_exactly_the_outside(fill, esize):
    rng = np.random.default_rng(11 + fill)
    dims, box = [21, 9, 3], [8, 4, 2]
    buf, strides = rand_tensor(rng, esize, dims, 3)
    v = rng.standard_normal(buf.size)  # finite values: any NaN in the image is the fill
    buf[:] = {oracle.FILL_NAN_F16: lambda: v.astype(np.float16).view(np.uint16),
              oracle.FILL_NAN_BF16: lambda: (v.astype(np.float32).view(np.uint32) >> 16)
              .astype(np.uint16),
              oracle.FILL_NAN_F32: lambda: v.astype(np.float32).view(np.uint32),
              oracle.FILL_NAN_F64: lambda: v.view(np.uint64)}[fill]()
    buf[::7] = 0  # in-bounds zeros must stay zeros
    view = strided_view(buf, 0, esize, dims, strides)
    for es in ([1, 1, 1], [3, 2, 1]):
        m = oracle.Map(buf, esize, dims, strides, box, estrides=es, fill=fill)
        mz = oracle.Map(buf, esize, dims, strides, box, estrides=es)
        for start in ([16, 8, 2], [-5, -2, 0], [0, 0, 0]):
            got = oracle.image(m, start).view(NP_UINT[esize])
            want, ok = box_stepped(view, start, box, es)
            ok = ok.reshape(-1)
            np.testing.assert_array_equal(got[ok], want.reshape(-1)[ok])
            assert np.isnan(as_float(got[~ok], fill)).all()
            assert not np.isnan(as_float(got[ok], fill)).any()
            np.testing.assert_array_equal(oracle.image(mz, start).view(NP_UINT[esize])[~ok], 0)


def test_nan_fill_keeps_whole_elements_under_swizzle_and_does_not_store():
    rng = np.random.default_rng(5)
    dims, box = [32, 10], [32, 8]
    buf, strides = rand_tensor(rng, 4, dims, 0)
    m = oracle.Map(buf, 4, dims, strides, box, fill=oracle.FILL_NAN_F32)
    ms = oracle.Map(buf, 4, dims, strides, box, span=128, fill=oracle.FILL_NAN_F32)
    none = oracle.image(m, [0, 8])
    np.testing.assert_array_equal(oracle.image(ms, [0, 8]), apply_page_swizzle128(none))
    assert np.isnan(none.view(np.float32)[64:]).all()  # rows 10..15 are outside
    before = buf.copy()
    oracle.store(m, [0, 8], none)
    np.testing.assert_array_equal(buf, before)  # only in-bounds elements written, unchanged


@pytest.mark.parametrize("kw", [dict(estrides=[0, 1]), dict(estrides=[9, 1]),
                                dict(estrides=[2, 1], span=128), dict(fill=oracle.FILL_NAN_F16),
                                dict(fill=oracle.FILL_NAN_F64), dict(fill=9)])
def test_undefined_maps_are_refused(kw):
    buf = np.zeros(64 * 4, np.uint32)
    span = kw.pop("span", 0)
    with pytest.raises(ValueError):
        oracle.Map(buf, 4, [32, 4], [256], [32, 4], span=span, **kw)
