"""GPU parity of two descriptor features against the oracle, through the C ABI:

- elementStrides (fangpin "gpu-hpc-book" ch. 08 "Cuda TMA", §"Tensor descriptor：CUtensorMap":
  the step, in elements, between the elements taken along each dim): copies on the tensor-map path
  (innermost step 1) and on the vector path (innermost step above 1, unaligned layouts, forced
  fallback, box lists off the 16-byte grid), round trips (always the vector path), and the
  allocation-free copy.  Bit-exact.
- NaN out-of-bounds fill (coolgpu "H200 · TMA · Tensor Memory Accelerator" §02): in-bounds image
  bytes equal the oracle's; out-of-bounds elements are NaN (any NaN is a correct fill).
"""
import numpy as np
import pytest

import oracle
from gpu_util import (ESIZE, as_float, assert_nan_fill, dev_map, guarded, host_map, to_dev,
                      to_host)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

U = {1: np.uint8, 2: np.uint16, 4: np.uint32, 8: np.uint64}


@pytest.fixture(scope="module")
def tm():
    import async_bulk_tensor_tmap_gb300 as m  # raises if the CUDA library is missing
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def check(tm):
    torch.cuda.synchronize()
    rc = tm.tm_stream_check()
    assert rc == tm.TM_OK, tm.tm_last_error()


def tensor(esize, dims, pitch_bytes, seed):
    """Random bytes for a tensor whose dim-0 rows are pitch_bytes apart (outer dims packed)."""
    rng = np.random.default_rng(seed)
    outer = int(np.prod(dims[1:])) if len(dims) > 1 else 1
    buf = rng.integers(0, 256, pitch_bytes * outer + 64, dtype=np.uint64).astype(np.uint8)
    strides, acc = [], pitch_bytes
    for d in dims[1:]:
        strides.append(acc)
        acc *= d
    return buf, strides


# name: (esize, dims, dim-0 pitch in bytes, box, elementStrides, span)
CASES = {
    "bf16_rows2_128B": (2, [128, 300], 256, [64, 32], [1, 2], 128),
    "bf16_cols2": (2, [200, 50], 448, [64, 16], [2, 1], 0),
    "f32_rank3_4_3_2": (4, [100, 20, 7], 400, [32, 8, 4], [4, 3, 2], 0),
    "u8_cols8": (1, [1000, 9], 1024, [128, 4], [8, 1], 0),
    "f64_rank5": (8, [10, 5, 4, 3, 2], 96, [4, 2, 3, 2, 1], [2, 1, 2, 2, 1], 0),
    "u16_3_5": (2, [96, 70], 192, [48, 16], [3, 5], 0),
    "bf16_rows3_64B": (2, [64, 33], 128, [32, 16], [1, 3], 64),
    "bf16_rows2_unaligned_pitch": (2, [120, 40], 250, [64, 8], [1, 2], 0),
    "f32_cols3_unaligned_pitch": (4, [50, 12], 212, [24, 4], [3, 2], 0),
    # every other element of 4-byte rows on a 16-byte pitch (the step-2 fast path; ragged last box)
    "f32_cols2": (4, [130, 20], 528, [32, 8], [2, 1], 0),
    # every other element of 2-byte rows whose starts are off 16 bytes (the general gather)
    "bf16_cols2_unaligned_pitch": (2, [200, 30], 418, [64, 8], [2, 1], 0),
}


def recipe(name):
    es, dims, pitch, box, steps, span = CASES[name]
    return es, dims, pitch, dict(box=box, estrides=steps, span=span, esize=es, dims=dims)


def setup_case(tm, name, seed=1):
    es, dims, pitch, r = recipe(name)
    buf, strides = tensor(es, dims, pitch, seed)
    r["strides"] = strides
    return buf, r


@pytest.mark.parametrize("force_fb", [False, True])
@pytest.mark.parametrize("name", sorted(CASES))
def test_strided_grid_copy(tm, name, force_fb):
    buf, r = setup_case(tm, name)
    m = dev_map(tm, to_dev(buf), r)
    aligned = "unaligned" not in name
    # a map whose innermost step is not 1 is routed to the vector path (TM_WHY_STEP0)
    tma = aligned and r["estrides"][0] == 1
    assert m.path == (tm.TM_PATH_TMA if tma else tm.TM_PATH_FALLBACK)
    assert bool(m.why_fallback & tm.TM_WHY_STEP0) == (r["estrides"][0] != 1)
    if force_fb:
        tm.tmap_force_fallback(m)
    om = host_map(buf, r)
    assert m.box_bytes == om.box_bytes and m.num_boxes == om.num_boxes
    imgs = guarded(m.num_boxes * m.box_bytes, 0x5A)
    tm.tiled_copy(m, None, imgs)
    check(tm)
    np.testing.assert_array_equal(to_host(imgs), oracle.tiled_copy(om))


@pytest.mark.parametrize("name", ["bf16_cols2", "f32_rank3_4_3_2", "u16_3_5", "bf16_rows2_128B"])
def test_strided_box_list(tm, name):
    """Starts off the box grid: negative, past the end, off the 16-byte grid (vector path) and on
    it (tensor-map path), more boxes than travel inline."""
    buf, r = setup_case(tm, name, seed=2)
    m = dev_map(tm, to_dev(buf), r)
    om = host_map(buf, r)
    rng = np.random.default_rng(3)
    rank = len(r["dims"])
    for aligned in (True, False):
        coords = []
        for _ in range(11):
            c = [int(rng.integers(-r["box"][i] + 1, r["dims"][i])) for i in range(rank)]
            if aligned:
                q = 16 // r["esize"]
                c[0] = c[0] // q * q
            coords.append(c)
        imgs = guarded(len(coords) * m.box_bytes, 0)
        tm.tiled_copy(m, coords, imgs)
        check(tm)
        np.testing.assert_array_equal(to_host(imgs), oracle.tiled_copy(om, coords=coords),
                                      err_msg=f"aligned={aligned}")


@pytest.mark.parametrize("name", sorted(CASES))
def test_strided_roundtrip_writes_exactly_the_taken_positions(tm, name):
    buf, r = setup_case(tm, name, seed=4)
    om = host_map(buf, r)
    rng = np.random.default_rng(5)
    imgs = rng.integers(0, 256, om.num_boxes * om.box_bytes, dtype=np.uint64).astype(np.uint8)
    dst = np.full_like(buf, 0xC3)
    dd = to_dev(dst)
    tm.tiled_roundtrip(dev_map(tm, dd, r), None, to_dev(imgs))
    check(tm)
    oracle.tiled_roundtrip(host_map(dst, r), imgs)
    np.testing.assert_array_equal(to_host(dd), dst)


@pytest.mark.parametrize("name", ["bf16_cols2", "f64_rank5", "bf16_rows2_128B"])
def test_strided_noalloc_copy(tm, name):
    buf, r = setup_case(tm, name, seed=6)
    m = dev_map(tm, to_dev(buf), r)
    om = host_map(buf, r)
    imgs = guarded(m.num_boxes * m.box_bytes, 0)
    tm.tiled_copy_noalloc(m, None, imgs)
    np.testing.assert_array_equal(to_host(imgs), oracle.tiled_copy(om))
    coords = [[-2, 1] + [0] * (len(r["dims"]) - 2), [3, -1] + [1] * (len(r["dims"]) - 2)]
    imgs2 = guarded(2 * m.box_bytes, 0)
    tm.tiled_copy_noalloc(m, coords, imgs2)
    np.testing.assert_array_equal(to_host(imgs2), oracle.tiled_copy(om, coords=coords))


# ---- NaN fill ----------------------------------------------------------------------------------
def finite_floats(dtype, tm, n, seed):
    v = np.random.default_rng(seed).standard_normal(n)
    if dtype == tm.TM_F16:
        return v.astype(np.float16).view(np.uint8)
    if dtype == tm.TM_BF16:
        return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16).view(np.uint8)
    if dtype == tm.TM_F32:
        return v.astype(np.float32).view(np.uint8)
    return v.view(np.uint8)




def nan_recipe(dtype, span, steps, cut=5):
    es = ESIZE[dtype]
    box0 = span // es if span else 64 // es
    dims = [3 * box0 - cut, 37, 3]
    pitch = (dims[0] * es + 15) // 16 * 16
    return dict(esize=es, dims=dims, strides=[pitch, pitch * 37], box=[box0, 8, 2], span=span,
                estrides=steps, nan=True)


@pytest.mark.parametrize("force_fb", [False, True])
@pytest.mark.parametrize("steps", [None, [1, 3, 2]])
@pytest.mark.parametrize("span", [0, 128])
@pytest.mark.parametrize("dt_name", ["TM_F16", "TM_BF16", "TM_F32", "TM_F64"])
def test_nan_fill_copy(tm, dt_name, span, steps, force_fb):
    dtype = getattr(tm, dt_name)
    r = nan_recipe(dtype, span, steps)
    n = r["strides"][1] * 3 // r["esize"]
    buf = finite_floats(dtype, tm, n, seed=7 + dtype)
    m = dev_map(tm, to_dev(buf), r, dtype=dtype)
    assert m.path == tm.TM_PATH_TMA
    if force_fb:
        tm.tmap_force_fallback(m)
    imgs = guarded(m.num_boxes * m.box_bytes, 0)
    tm.tiled_copy(m, None, imgs)
    check(tm)
    want = oracle.tiled_copy(host_map(buf, r, dtype=dtype))
    assert_nan_fill(to_host(imgs), want, dtype, tm)


@pytest.mark.parametrize("dt_name", ["TM_F16", "TM_BF16", "TM_F32", "TM_F64"])
def test_nan_fill_pattern_same_on_both_paths(tm, dt_name):
    """The vector path writes the NaN bit pattern the tensor-map hardware writes."""
    dtype = getattr(tm, dt_name)
    r = nan_recipe(dtype, 0, None)
    n = r["strides"][1] * 3 // r["esize"]
    buf = finite_floats(dtype, tm, n, seed=9)
    bd = to_dev(buf)
    outs = []
    for force_fb in (False, True):
        m = dev_map(tm, bd, r, dtype=dtype)
        if force_fb:
            tm.tmap_force_fallback(m)
        imgs = guarded(m.num_boxes * m.box_bytes, 0)
        q = 16 // r["esize"]  # starts on the 16-byte grid: the tensor-map path takes the list
        tm.tiled_copy(m, [[-q, -1, 0], [(r["dims"][0] - 3) // q * q, 30, 2]], imgs)
        check(tm)
        outs.append(to_host(imgs).view(U[r["esize"]]))
    hw = sorted({hex(int(v)) for v in outs[0][np.isnan(as_float(outs[0], dtype, tm))]})
    print(f"{dt_name} NaN fill written by the tensor-map path: {hw}")
    np.testing.assert_array_equal(outs[1], outs[0])


@pytest.mark.parametrize("cut", [4, 5])  # row of 368 bytes: tensor store / reduce; 364: vector
def test_nan_fill_map_stores_and_reduces_in_bounds_only(tm, cut):
    """The fill never reaches memory: a round trip and a reduce through NaN-fill maps change no
    out-of-bounds byte, and their in-bounds results equal the oracle's."""
    dtype = tm.TM_F32
    r = nan_recipe(dtype, 128, None, cut)
    n = r["strides"][1] * 3 // 4
    src = finite_floats(dtype, tm, n, seed=11)
    dst = finite_floats(dtype, tm, n, seed=12)
    sd, dd = to_dev(src), to_dev(dst)
    tm.tile_reduce(dev_map(tm, dd, r, dtype=dtype), dev_map(tm, sd, r, dtype=dtype), tm.TM_RED_ADD)
    check(tm)
    oracle.tile_reduce(host_map(dst, r, dtype=dtype), host_map(src, r, dtype=dtype), oracle.F32,
                       oracle.ADD)
    np.testing.assert_array_equal(to_host(dd), dst)
    m = dev_map(tm, sd, r, dtype=dtype)
    imgs = guarded(m.num_boxes * m.box_bytes, 0)
    tm.tiled_copy(m, None, imgs)
    out = np.full_like(src, 0x3C)
    od = to_dev(out)
    tm.tiled_roundtrip(dev_map(tm, od, r, dtype=dtype), None, imgs)
    check(tm)
    oracle.tiled_roundtrip(host_map(out, r, dtype=dtype), oracle.tiled_copy(host_map(src, r,
                                                                                     dtype=dtype)))
    np.testing.assert_array_equal(to_host(od), out)
