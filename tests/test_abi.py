"""The C-ABI library without a GPU: it loads, exports every call include/tmap.h declares, and its
host-side logic (validation, path choice, box grid) follows the constraint table of the coolgpu
"H200 · TMA · Tensor Memory Accelerator" card §03 and the swizzle rules of mlc.ai "Modern GPU
Programming for MLSys", chapter "异步数据搬运：TMA".  No kernel is launched here."""
import ctypes
import os
import re

import pytest

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tmap.h")


@pytest.fixture(scope="module")
def tm():
    import __graft_entry__
    __graft_entry__._cuda_build_module().build()
    import async_bulk_tensor_tmap_gb300 as m
    return m


FAKE = 1 << 24  # a 16-byte aligned stand-in address; tmap_plan never dereferences it


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(\w+)\s*\(", text, re.M)))


def test_library_exports_every_declared_call(tm):
    names = declared_functions()
    assert {"tmap_encode", "tile_load_image", "tiled_copy", "tiled_roundtrip", "tile_reduce_add",
            "stream_tiles"} <= set(names)
    lib = ctypes.CDLL(tm.library_path)
    for n in names:
        assert hasattr(lib, n), n


def test_package_refuses_to_import_without_the_library(tmp_path):
    """No CPU fallback: a copy of the package without its CUDA library fails at import."""
    import shutil
    import subprocess
    import sys
    pkg = tmp_path / "async_bulk_tensor_tmap_gb300"
    pkg.mkdir()
    shutil.copy(os.path.join(ROOT, "async_bulk_tensor_tmap_gb300", "__init__.py"), pkg)
    r = subprocess.run([sys.executable, "-c", "import async_bulk_tensor_tmap_gb300"],
                       cwd=tmp_path, capture_output=True, text=True)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "is missing" in r.stderr


def test_desc_layout(tm):
    assert tm._L.tm_desc_size() == 384
    m = tm.TensorMap()
    assert m.ptr % 64 == 0


def plan(tm, **kw):
    args = dict(dtype=tm.TM_BF16, base=FAKE, global_dim=[8192, 8192], global_strides=[16384],
                box_dim=[64, 128], swizzle=tm.TM_SWIZZLE_128B)
    args.update(kw)
    return tm.tmap_plan(**args)


def code_of(tm, **kw):
    try:
        plan(tm, **kw)
    except tm.TmapError as e:
        return e.code
    return tm.TM_OK


def test_plan_w3_grid(tm):
    m = plan(tm)
    assert (m.box_bytes, m.num_boxes, m.path) == (16384, 8192, tm.TM_PATH_TMA)


def test_plan_rejections(tm):
    assert code_of(tm, global_dim=[8] * 6, global_strides=[16] * 5, box_dim=[8] * 6,
                   swizzle=0) == tm.TM_EINVAL                                     # rank > 5
    assert code_of(tm, box_dim=[64, 257]) == tm.TM_ERANGE                          # box > 256
    assert code_of(tm, box_dim=[64, 0]) == tm.TM_ERANGE
    assert code_of(tm, global_dim=[0, 8]) == tm.TM_ERANGE
    assert code_of(tm, global_dim=[(1 << 32) + 1, 8]) == tm.TM_ERANGE
    assert code_of(tm, box_dim=[60, 8], swizzle=0) == tm.TM_EALIGN                 # 120 B inner
    assert code_of(tm, box_dim=[32, 8]) == tm.TM_EUNSUPPORTED                      # 64 B != 128B
    assert code_of(tm, box_dim=[128, 8]) == tm.TM_EUNSUPPORTED                     # 256 B > atom
    assert code_of(tm, global_strides=[1 << 40]) == tm.TM_ERANGE                   # stride >= 2^40
    assert code_of(tm, global_strides=[16383]) == tm.TM_EALIGN                     # not % esize
    assert code_of(tm, base=FAKE + 1) == tm.TM_EALIGN
    assert code_of(tm, element_strides=[2, 1]) == tm.TM_EUNSUPPORTED              # swizzled
    assert code_of(tm, element_strides=[1, 9]) == tm.TM_EINVAL
    assert code_of(tm, element_strides=[1, 0]) == tm.TM_EINVAL
    assert code_of(tm, element_strides=[3, 1], swizzle=0) == tm.TM_EALIGN  # 22 * 2 B image row
    assert code_of(tm, oob=tm.TM_OOB_NAN, dtype=tm.TM_U16) == tm.TM_EINVAL
    assert code_of(tm, oob=2) == tm.TM_EINVAL
    assert code_of(tm, dtype=42) == tm.TM_EINVAL
    assert code_of(tm, base=0) == tm.TM_EINVAL
    assert code_of(tm, box_dim=[256, 256, 4], global_dim=[256, 256, 4],
                   global_strides=[512, 512 * 256], swizzle=0) == tm.TM_ERANGE     # 512 KiB box


def test_plan_routes_unaligned_layouts_to_fallback(tm):
    r5 = workloads.w4_rank5_map()
    m = tm.tmap_plan(tm.TM_BF16, FAKE, r5["dims"], r5["strides"], r5["box"])
    assert m.path == tm.TM_PATH_FALLBACK and m.why_fallback == tm.TM_WHY_STRIDE
    assert (m.box_bytes, m.num_boxes) == (40960, 4096)
    m = plan(tm, base=FAKE + 8)
    assert m.path == tm.TM_PATH_FALLBACK and m.why_fallback == tm.TM_WHY_BASE


@pytest.mark.parametrize("box_cols,span,boxes", [(64, 128, 16384), (32, 64, 32768)])
def test_plan_w4_rank3_grids(tm, box_cols, span, boxes):
    r = workloads.w4_rank3_map(box_cols, span=span)
    sw = {128: tm.TM_SWIZZLE_128B, 64: tm.TM_SWIZZLE_64B}[span]
    m = tm.tmap_plan(tm.TM_BF16, FAKE, r["dims"], r["strides"], r["box"], swizzle=sw)
    assert (m.path, m.num_boxes) == (tm.TM_PATH_TMA, boxes)


def test_plan_w5_grids(tm):
    r = workloads.w5a_map()
    m = tm.tmap_plan(tm.TM_F32, FAKE, r["dims"], r["strides"], r["box"], swizzle=3)
    assert (m.num_boxes, m.box_bytes) == (65536, 16384)
    a, b = workloads.w5b_maps()
    ma = tm.tmap_plan(tm.TM_BF16, FAKE, a["dims"], a["strides"], a["box"], swizzle=3)
    mb = tm.tmap_plan(tm.TM_BF16, FAKE, b["dims"], b["strides"], b["box"], swizzle=3)
    assert ma.num_boxes == mb.num_boxes == 4096
    assert ma.box_bytes + mb.box_bytes == 32768


def test_plan_w2_regroup_views(tm):
    m = tm.tmap_plan(tm.TM_F16, FAKE, [64, 16, 4], [512, 128], [64, 16, 2], swizzle=3)
    assert (m.path, m.num_boxes, m.box_bytes) == (tm.TM_PATH_TMA, 2, 4096)
    m = tm.tmap_plan(tm.TM_F16, FAKE, [32, 16, 8], [512, 64], [32, 16, 4], swizzle=2)
    assert (m.path, m.num_boxes, m.box_bytes) == (tm.TM_PATH_TMA, 2, 4096)
    m = tm.tmap_plan(tm.TM_F16, FAKE, [16, 16, 16], [512, 32], [16, 16, 8], swizzle=1)
    assert (m.path, m.num_boxes, m.box_bytes) == (tm.TM_PATH_TMA, 2, 4096)


def test_force_fallback_flag(tm):
    m = plan(tm)
    tm.tmap_force_fallback(m)
    assert m.path == tm.TM_PATH_FALLBACK and m.why_fallback & tm.TM_WHY_FORCED


def test_pick_swizzle(tm):
    assert [tm.tm_pick_swizzle(x) for x in (128, 64, 32, 16, 256)] == [
        tm.TM_SWIZZLE_128B, tm.TM_SWIZZLE_64B, tm.TM_SWIZZLE_32B, tm.TM_SWIZZLE_NONE,
        tm.TM_SWIZZLE_NONE]


def test_calls_reject_unfilled_descriptors(tm):
    blank = tm.TensorMap()
    with pytest.raises(tm.TmapError) as e:
        tm.tiled_copy(blank, None, FAKE, stream=0)
    assert e.value.code == tm.TM_EINVAL
    m = plan(tm)
    with pytest.raises(tm.TmapError) as e:
        tm.tiled_copy(m, None, FAKE + 8, stream=0)
    assert e.value.code == tm.TM_EALIGN
    with pytest.raises(tm.TmapError) as e:
        tm.stream_tiles(m, m, 1, FAKE, FAKE, FAKE, FAKE, stream=0)
    assert e.value.code == tm.TM_ERANGE


def test_empty_box_list_is_a_no_op(tm):
    """An empty box list (coords given, nbox 0) returns at once without touching the device, so
    it needs no image buffer; a non-empty list still needs one."""
    m = plan(tm)
    tm.tiled_copy(m, [], None, stream=0)
    tm.tiled_roundtrip(m, [], None, stream=0)
    tm.tiled_copy_noalloc(m, [], None, stream=0)
    for call in (tm.tiled_copy, tm.tiled_roundtrip, tm.tiled_copy_noalloc):
        with pytest.raises(tm.TmapError) as e:
            call(m, [[0, 0]], None, stream=0)
        assert e.value.code == tm.TM_EINVAL
    with pytest.raises(tm.TmapError) as e:  # the whole grid is never empty
        tm.tiled_copy(m, None, None, stream=0)
    assert e.value.code == tm.TM_EINVAL


def test_plan_element_strides_and_nan_fill(tm):
    """Image extents are ceil(box / elementStrides); the box grid keeps stepping by the box."""
    m = plan(tm, element_strides=[1, 3], oob=tm.TM_OOB_NAN)
    assert (m.box_bytes, m.num_boxes, m.path) == (128 * 43, 8192, tm.TM_PATH_TMA)
    assert list(m.d.estride[:2]) == [1, 3] and m.d.oob == tm.TM_OOB_NAN
    m = plan(tm, element_strides=[2, 8], box_dim=[128, 16], swizzle=0)
    assert (m.box_bytes, m.num_boxes) == (64 * 2 * 2, 64 * 512)
    assert (m.path, m.why_fallback) == (tm.TM_PATH_FALLBACK, tm.TM_WHY_STEP0)
    for dt in (tm.TM_F16, tm.TM_BF16, tm.TM_F32, tm.TM_F64):
        assert code_of(tm, dtype=dt, box_dim=[64 if dt in (tm.TM_F16, tm.TM_BF16) else
                                             (32 if dt == tm.TM_F32 else 16), 8],
                       oob=tm.TM_OOB_NAN) == tm.TM_OK


def test_reduce_and_ring_refuse_strided_or_nan_maps(tm):
    """Checked on the host before any device work (so this runs without a GPU)."""
    f = dict(dtype=tm.TM_F32, box_dim=[32, 128])
    a = plan(tm, **f)
    s = plan(tm, element_strides=[1, 2], **f)
    for dst, src in ((a, s), (s, a)):
        with pytest.raises(tm.TmapError) as e:
            tm.tile_reduce(dst, src, tm.TM_RED_ADD, stream=0)
        assert e.value.code == tm.TM_EUNSUPPORTED
    ring = dict(box_dim=[64, 128])
    ok, nan, step = plan(tm, **ring), plan(tm, oob=tm.TM_OOB_NAN, **ring), \
        plan(tm, element_strides=[1, 2], **ring)
    out = 1 << 41  # never dereferenced: the call fails validation first
    for x, y in ((ok, nan), (step, ok)):
        with pytest.raises(tm.TmapError) as e:
            tm.stream_tiles(x, y, 4, out, out, out, out, stream=0)
        assert e.value.code == tm.TM_EUNSUPPORTED


def test_stream_gemm_validation(tm):
    """Checked on the host before any device work (so this runs without a GPU)."""
    a = tm.tmap_plan(tm.TM_BF16, FAKE, [4096, 512], [8192], [64, 128], swizzle=tm.TM_SWIZZLE_128B)
    b = tm.tmap_plan(tm.TM_BF16, FAKE, [4096, 768], [8192], [64, 256], swizzle=tm.TM_SWIZZLE_128B)
    c = 1 << 41  # never dereferenced: every case below fails validation first

    def code(*args, **kw):
        try:
            tm.stream_gemm(*args, stream=0, **kw)
        except tm.TmapError as e:
            return e.code
        return tm.TM_OK

    assert code(b, a, c) == tm.TM_EUNSUPPORTED                    # boxes swapped
    assert code(a, b, c, stages=1) == tm.TM_ERANGE
    assert code(a, b, c, stages=8) == tm.TM_ERANGE
    assert code(a, b, c, ldc=700) == tm.TM_EINVAL                 # ldc < N
    assert code(a, b, c + 8) == tm.TM_EALIGN
    assert code(a, b, c, ldc=770) == tm.TM_EALIGN
    b2 = tm.tmap_plan(tm.TM_BF16, FAKE, [4032, 768], [8192], [64, 256], swizzle=tm.TM_SWIZZLE_128B)
    assert code(a, b2, c) == tm.TM_EINVAL                         # K differs
    f = tm.tmap_plan(tm.TM_F16, FAKE, [4096, 512], [8192], [64, 128], swizzle=tm.TM_SWIZZLE_128B)
    assert code(f, b, c) == tm.TM_EUNSUPPORTED
    n = tm.tmap_plan(tm.TM_BF16, FAKE, [4096, 512], [8192], [64, 128])
    assert code(n, b, c) == tm.TM_EUNSUPPORTED                    # no swizzle


def test_l2_promotion_field(tm, monkeypatch):
    """The map's L2 promotion: 128B unless TM_L2_PROMOTION says otherwise, set per map, values
    above TM_L2_256B and unfilled descriptors refused (no GPU: a planned map keeps the value for a
    later encode)."""
    monkeypatch.delenv("TM_L2_PROMOTION", raising=False)
    m = plan(tm)
    assert m.l2_promotion == tm.TM_L2_128B
    for p in (tm.TM_L2_NONE, tm.TM_L2_64B, tm.TM_L2_256B):
        tm.tmap_set_l2_promotion(m, p)
        assert m.l2_promotion == p
    with pytest.raises(tm.TmapError) as e:
        tm.tmap_set_l2_promotion(m, 4)
    assert e.value.code == tm.TM_EINVAL
    with pytest.raises(tm.TmapError) as e:
        tm.tmap_set_l2_promotion(tm.TensorMap(), tm.TM_L2_NONE)
    assert e.value.code == tm.TM_EINVAL
    monkeypatch.setenv("TM_L2_PROMOTION", "0")
    assert plan(tm).l2_promotion == tm.TM_L2_NONE
