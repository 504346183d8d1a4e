"""GPU parity of the general reduce (tile_reduce): add / min / max over f32, f16, bf16, u32 and
s32, on the bulk tensor reduce and on the vector path, bit for bit against the oracle
(fangpin "gpu-hpc-book" ch. 08 "Cuda TMA", §"TMA reduce，把“搬运”和“归约”合并")."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import host_map, to_dev, to_host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

KINDS = ["f32", "f16", "bf16", "u32", "s32"]
ORC_TYPE = {"f32": oracle.F32, "f16": oracle.F16, "bf16": oracle.BF16, "u32": oracle.U32,
            "s32": oracle.S32}


@pytest.fixture(scope="module")
def tm():
    import async_bulk_tensor_tmap_gb300 as m  # raises if the CUDA library is missing
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def tm_dtype(tm, kind):
    return {"f32": tm.TM_F32, "f16": tm.TM_F16, "bf16": tm.TM_BF16, "u32": tm.TM_U32,
            "s32": tm.TM_S32}[kind]


def recipe(kind, rows, cols, pitch):
    es = 2 if kind in ("f16", "bf16") else 4
    return dict(dims=[cols, rows], strides=[pitch * es], box=[128 // es, 128], span=128, esize=es)


def run_case(tm, kind, op, rows, cols, pitch, force_fallback, seed):
    d, s = workloads.reduce_operands(kind, rows, pitch, seed)
    r = recipe(kind, rows, cols, pitch)
    dd, sd = to_dev(d), to_dev(s)
    dt = tm_dtype(tm, kind)
    md = tm.tmap_encode(dt, dd, r["dims"], r["strides"], r["box"], swizzle=tm.TM_SWIZZLE_128B)
    ms = tm.tmap_encode(dt, sd, r["dims"], r["strides"], r["box"], swizzle=tm.TM_SWIZZLE_128B)
    if force_fallback:
        tm.tmap_force_fallback(md)
    tm.tile_reduce(md, ms, op)
    torch.cuda.synchronize()
    assert tm.tm_stream_check() == tm.TM_OK, tm.tm_last_error()
    hd = np.ascontiguousarray(d).copy()
    oracle.tile_reduce(host_map(hd, r), host_map(np.ascontiguousarray(s), r), ORC_TYPE[kind], op)
    got = to_host(dd)
    np.testing.assert_array_equal(got, hd.reshape(-1).view(np.uint8),
                                  err_msg=f"{kind} op {op} fallback={force_fallback}")


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("op", [0, 1, 2])
@pytest.mark.parametrize("force_fallback", [False, True])
def test_reduce_ops(tm, kind, op, force_fallback):
    # 300 x 200 in bounds (ragged in both dims), padding columns up to 208 must stay untouched
    run_case(tm, kind, op, 300, 200, 208, force_fallback, seed=100 + 7 * op + KINDS.index(kind))


def _nan_mask(bits, kind):
    b = bits.astype(np.uint32)
    if kind == "f32":
        return ((b & 0x7F800000) == 0x7F800000) & ((b & 0x007FFFFF) != 0)
    if kind == "f16":
        return ((b & 0x7C00) == 0x7C00) & ((b & 0x03FF) != 0)
    if kind == "bf16":
        return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)
    return np.zeros(b.shape, bool)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("op", [0, 1, 2])
@pytest.mark.parametrize("force_fallback", [False, True])
def test_reduce_special_values(tm, kind, op, force_fallback):
    """Every pair of the formats' special values (zeros of both signs, subnormals, the smallest
    normal, the largest finite, infinities, NaNs; integer wrap points) and a seeded mix around
    them, on the bulk tensor reduce and on the vector path.  Bit for bit against the oracle where
    its result is a number; where it is a NaN, a NaN (the payload of an operation's NaN is open)."""
    rows, cols, pitch = 64, 96, 96
    d, s = workloads.special_reduce_operands(kind, rows, pitch, seed=500 + 3 * op + KINDS.index(kind))
    r = recipe(kind, rows, cols, pitch)
    dd, sd = to_dev(d), to_dev(s)
    dt = tm_dtype(tm, kind)
    md = tm.tmap_encode(dt, dd, r["dims"], r["strides"], r["box"], swizzle=tm.TM_SWIZZLE_128B)
    ms = tm.tmap_encode(dt, sd, r["dims"], r["strides"], r["box"], swizzle=tm.TM_SWIZZLE_128B)
    if force_fallback:
        tm.tmap_force_fallback(md)
    tm.tile_reduce(md, ms, op)
    torch.cuda.synchronize()
    assert tm.tm_stream_check() == tm.TM_OK, tm.tm_last_error()
    hd = np.ascontiguousarray(d).copy()
    oracle.tile_reduce(host_map(hd, r), host_map(np.ascontiguousarray(s), r), ORC_TYPE[kind], op)
    es = r["esize"]
    ut = np.uint32 if es == 4 else np.uint16
    want = hd.reshape(-1).view(ut)
    got = to_host(dd).view(ut)
    nan = _nan_mask(want, kind)
    bad = np.flatnonzero(~nan & (got != want))
    assert bad.size == 0, (f"{kind} op {op} fallback={force_fallback}: {bad.size} mismatches, first "
                           f"dst {d.reshape(-1).view(ut)[bad[0]]:#x} src {s.reshape(-1).view(ut)[bad[0]]:#x} "
                           f"got {got[bad[0]]:#x} want {want[bad[0]]:#x}")
    assert _nan_mask(got[nan], kind).all(), f"{kind} op {op}: a NaN result came back as a number"


@pytest.mark.parametrize("kind", ["bf16", "u32"])
def test_reduce_ragged_row_end_keeps_padding(tm, kind):
    # inner extent not a multiple of 16 bytes: the vector path, padding must survive
    run_case(tm, kind, 0, 130, 99, 104, False, seed=300)


def test_reduce_rejects_mixed_types(tm):
    d = torch.zeros(64 * 64 * 4, dtype=torch.uint8, device="cuda")
    a = tm.tmap_encode(tm.TM_F32, d, [64, 64], [256], [32, 64], swizzle=tm.TM_SWIZZLE_128B)
    b = tm.tmap_encode(tm.TM_U32, d, [64, 64], [256], [32, 64], swizzle=tm.TM_SWIZZLE_128B)
    with pytest.raises(tm.TmapError) as e:
        tm.tile_reduce(a, b, tm.TM_RED_ADD)
    assert e.value.code == tm.TM_EINVAL
    c = tm.tmap_encode(tm.TM_U8, d, [256, 64], [256], [128, 64], swizzle=tm.TM_SWIZZLE_128B)
    with pytest.raises(tm.TmapError) as e:
        tm.tile_reduce(c, c, tm.TM_RED_MAX)
    assert e.value.code == tm.TM_EUNSUPPORTED


# Views whose two innermost dims are contiguous (a row split into G groups of c0 elements, the
# group stride c0 * esize not a multiple of 16: the vector path, which walks such a view by whole
# rows), ragged boxes along every dim, padding after each row that must stay untouched; `shifted`
# moves the destination one element along so that the two tensors' 16-byte phases differ (the
# element-by-element path); `src_gaps` gives the source a gap between groups (no fusion).
@pytest.mark.parametrize("kind,op,c0", [("bf16", 0, 60), ("f16", 0, 60), ("f32", 2, 50),
                                        ("s32", 1, 50)])
@pytest.mark.parametrize("layout", ["same", "shifted", "src_gaps"])
def test_reduce_unaligned_view_by_rows(tm, kind, op, c0, layout):
    es = 2 if kind in ("f16", "bf16") else 4
    R, G = 37, 5
    P = G * (c0 + 4) + 8  # row pitch in elements, room for the source's gaps and padding
    d, s = workloads.reduce_operands(kind, R, P, 400 + op + KINDS.index(kind))
    box = [64 // es, G, 8]
    rd = dict(dims=[c0, G, R], strides=[c0 * es, P * es], box=box, span=0, esize=es)
    rs = dict(rd, strides=[(c0 + 4) * es, P * es]) if layout == "src_gaps" else rd
    off = es if layout == "shifted" else 0
    dd, sd = to_dev(d), to_dev(s)
    dt = tm_dtype(tm, kind)
    md = tm.tmap_encode(dt, dd.data_ptr() + off, rd["dims"], rd["strides"], rd["box"])
    ms = tm.tmap_encode(dt, sd, rs["dims"], rs["strides"], rs["box"])
    assert md.path == tm.TM_PATH_FALLBACK
    tm.tile_reduce(md, ms, op)
    torch.cuda.synchronize()
    assert tm.tm_stream_check() == tm.TM_OK, tm.tm_last_error()
    hd = np.ascontiguousarray(d).copy()
    oracle.tile_reduce(host_map(hd, rd, offset=off), host_map(np.ascontiguousarray(s), rs),
                       ORC_TYPE[kind], op)
    np.testing.assert_array_equal(to_host(dd), hd.reshape(-1).view(np.uint8),
                                  err_msg=f"{kind} op {op} {layout}")
