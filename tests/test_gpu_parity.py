"""GPU parity: every result of the CUDA path, through the C ABI, equals the CPU oracle's bit for
bit, on the pages' example shapes and on reduced copies of the large workloads that still span
several boxes and a ragged tail.

Page tags: [MLSys-TMA] mlc.ai "Modern GPU Programming for MLSys", chapter "异步数据搬运：TMA";
[Book-TMA] fangpin "gpu-hpc-book" ch. 08 "Cuda TMA"; [H200-TMA] coolgpu H200 TMA feature card.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import (assert_nan_fill, dev_map, empty_images, full_like, guarded, host_map, to_dev,
                      to_host)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tm():
    import async_bulk_tensor_tmap_gb300 as m  # raises if the CUDA library is missing
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def check(tm):
    torch.cuda.synchronize()
    rc = tm.tm_stream_check()
    assert rc == tm.TM_OK, tm.tm_last_error()


def w1_recipe(span):
    return dict(dims=[128, 16], strides=[256], box=[64, 8], span=span, esize=2)


# ---- W1: [MLSys-TMA] §"TMA 如何写入 swizzled layout", 16 x 128 fp16, one 8 x 64 box --------------
@pytest.mark.parametrize("span", [0, 128])
@pytest.mark.parametrize("start", [(0, 0), (64, 8)])
def test_w1_image_and_roundtrip(tm, span, start):
    x = workloads.w1_tensor()
    r = w1_recipe(span)
    xd = to_dev(x)
    m = dev_map(tm, xd, r, dtype=tm.TM_F16)
    assert m.path == tm.TM_PATH_TMA
    img = empty_images(1, 1024)
    tm.tile_load_image(m, list(start), img)
    check(tm)
    want = oracle.image(host_map(x, r), start)
    np.testing.assert_array_equal(to_host(img), want)
    # round trip into a sentinel-filled tensor: only the box's elements change
    dst = guarded(16 * 128 * 2, 0xEE)
    md = dev_map(tm, dst, r, dtype=tm.TM_F16)
    tm.tiled_roundtrip(md, [list(start)], img)
    check(tm)
    host_dst = np.full(16 * 128 * 2, 0xEE, dtype=np.uint8)
    oracle.store(host_map(host_dst, r), start, want)
    np.testing.assert_array_equal(to_host(dst), host_dst)


# ---- W2: [MLSys-TMA] §"用 3D TMA 搬运多个 swizzle atoms", 3-D regrouped views --------------------
W2_VIEWS = {128: (64, [0, 0, 0], [0, 0, 2]), 64: (32, [0, 0, 0], [0, 0, 4]),
            32: (16, [0, 0, 0], [0, 0, 8])}


@pytest.mark.parametrize("span", [128, 64, 32])
def test_w2_regrouped_views(tm, span):
    x = workloads.w2_tensor()
    gcols, c0, c1 = W2_VIEWS[span]
    r = dict(dims=[gcols, 16, 256 // gcols], strides=[512, gcols * 2], box=[gcols, 16, 128 // gcols],
             span=span, esize=2)
    xd = to_dev(x)
    m = dev_map(tm, xd, r, dtype=tm.TM_F16)
    imgs = empty_images(2, 4096)
    tm.tiled_copy(m, [c0, c1], imgs)
    check(tm)
    want = oracle.tiled_copy(host_map(x, r), coords=[c0, c1])
    np.testing.assert_array_equal(to_host(imgs), want)
    print(f"W2 {span}B view path={m.path} why={m.why_fallback}")
    if span == 128:  # the per-slice map (base moved to column 128) gives the same second image
        rs = dict(dims=[64, 16, 2], strides=[512, 128], box=[64, 16, 2], span=128, esize=2)
        ms = dev_map(tm, xd, rs, offset=256, dtype=tm.TM_F16)
        one = empty_images(1, 4096)
        tm.tile_load_image(ms, [0, 0, 0], one)
        check(tm)
        np.testing.assert_array_equal(to_host(one), want[4096:])


# ---- W3 (reduced): bf16 matrix, 128 x 64 boxes, 128B, ragged in both dims -------------------------
def w3_small(span=128, rows=1000, cols=776):
    x = workloads.w3_tensor(rows, cols, seed=31)
    return x, workloads.w3_map(rows, cols, span=span)


@pytest.mark.parametrize("span", [128, 0])
@pytest.mark.parametrize("force_fallback", [False, True])
def test_w3_copy_and_roundtrip(tm, span, force_fallback):
    x, r = w3_small(span)
    xd = to_dev(x)
    m = dev_map(tm, xd, r)
    if force_fallback:
        tm.tmap_force_fallback(m)
    n, bb = m.num_boxes, m.box_bytes
    assert n == 8 * 13
    imgs = empty_images(n, bb)
    tm.tiled_copy(m, None, imgs)
    check(tm)
    want = oracle.tiled_copy(host_map(x, r), threads=8)
    np.testing.assert_array_equal(to_host(imgs), want)
    dst = full_like(xd, 0x77)
    md = dev_map(tm, dst, r)
    if force_fallback:
        tm.tmap_force_fallback(md)
    tm.tiled_roundtrip(md, None, imgs)
    check(tm)
    assert torch.equal(dst, xd)


def test_l2_promotion_changes_no_byte(tm):
    """Every L2 promotion of the tensor map gives the oracle's images, and a rebase keeps it."""
    x, r = w3_small(128, rows=520, cols=392)
    xd = to_dev(x)
    want = oracle.tiled_copy(host_map(x, r), threads=8)
    m = dev_map(tm, xd, r)
    for p in (tm.TM_L2_NONE, tm.TM_L2_64B, tm.TM_L2_128B, tm.TM_L2_256B):
        tm.tmap_set_l2_promotion(m, p)
        assert m.path == tm.TM_PATH_TMA and m.l2_promotion == p
        imgs = empty_images(m.num_boxes, m.box_bytes)
        tm.tiled_copy(m, None, imgs)
        check(tm)
        np.testing.assert_array_equal(to_host(imgs), want, err_msg=f"promotion {p}")
    x2 = to_dev(x)
    tm.tmap_replace_address(m, x2)
    assert m.l2_promotion == tm.TM_L2_256B
    imgs = empty_images(m.num_boxes, m.box_bytes)
    tm.tiled_copy(m, None, imgs)
    check(tm)
    np.testing.assert_array_equal(to_host(imgs), want)


# Small boxes share a stage, each in a slot starting on its swizzle period (1024 / 512 / 256 bytes
# for 128B / 64B / 32B, 128 without): padded slots (box smaller than its period) move one bulk copy
# per box; dense ones one per stage.  Copy, round trip and reduce-add on the tensor-map path.
@pytest.mark.parametrize("box,span", [([64, 4], 128), ([32, 4], 64), ([16, 4], 32), ([8, 3], 0),
                                      ([64, 8], 0), ([32, 8], 64)])
def test_small_boxes_share_stages(tm, box, span):
    x, r = w3_small(span, rows=203, cols=392)
    r = dict(r, box=box)
    xd = to_dev(x)
    m = dev_map(tm, xd, r)
    assert m.path == tm.TM_PATH_TMA and m.box_bytes == box[0] * box[1] * 2
    imgs = empty_images(m.num_boxes, m.box_bytes)
    tm.tiled_copy(m, None, imgs)
    check(tm)
    want = oracle.tiled_copy(host_map(x, r), threads=8)
    np.testing.assert_array_equal(to_host(imgs), want)
    dst = full_like(xd, 0x77)
    tm.tiled_roundtrip(dev_map(tm, dst, r), None, imgs)
    check(tm)
    assert torch.equal(dst, xd)


@pytest.mark.parametrize("box,span", [([32, 4], 128), ([4, 3], 0)])
def test_small_boxes_reduce_add(tm, box, span):
    d, s = workloads.w5a_tensors(rows=130, cols=96, seed_dst=15, seed_src=16)
    r = dict(workloads.w5a_map(rows=130, cols=96, span=span), box=box)
    dd, sd = to_dev(d), to_dev(s)
    md, ms = dev_map(tm, dd, r), dev_map(tm, sd, r)
    assert md.path == tm.TM_PATH_TMA
    tm.tile_reduce_add(md, ms)
    check(tm)
    hd = d.copy()
    oracle.tile_reduce_add(host_map(hd, r), host_map(s, r))
    np.testing.assert_array_equal(to_host(dd).view(np.uint32), hd.reshape(-1).view(np.uint32))


def test_w3_fallback_and_tma_images_identical(tm):
    x, r = w3_small(128, rows=520, cols=392)
    xd = to_dev(x)
    a, b = dev_map(tm, xd, r), dev_map(tm, xd, r)
    tm.tmap_force_fallback(b)
    ia, ib = empty_images(a.num_boxes, a.box_bytes, 1), empty_images(b.num_boxes, b.box_bytes, 2)
    tm.tiled_copy(a, None, ia)
    tm.tiled_copy(b, None, ib)
    check(tm)
    assert torch.equal(ia, ib)


def test_unaligned_base_takes_fallback(tm):
    x, r = w3_small(0, rows=300, cols=200)
    raw = np.zeros(x.size * 2 + 64, np.uint8)
    raw[8:8 + x.size * 2] = x.reshape(-1).view(np.uint8)
    rd = to_dev(raw)
    m = dev_map(tm, rd, r, offset=8)
    assert m.path == tm.TM_PATH_FALLBACK and m.why_fallback == tm.TM_WHY_BASE
    imgs = empty_images(m.num_boxes, m.box_bytes)
    tm.tiled_copy(m, None, imgs)
    check(tm)
    want = oracle.tiled_copy(host_map(raw, r, offset=8))
    np.testing.assert_array_equal(to_host(imgs), want)
    out = full_like(rd, 0x33)
    mo = dev_map(tm, out, r, offset=8)
    tm.tiled_roundtrip(mo, None, imgs)
    check(tm)
    host_out = np.full_like(raw, 0x33)
    oracle.tiled_roundtrip(host_map(host_out, r, offset=8), want)
    np.testing.assert_array_equal(to_host(out), host_out)


# ---- explicit box lists: inline (<= 8) and staged in device memory; odd starts go to fallback ---
@pytest.mark.parametrize("nbox", [5, 40])
@pytest.mark.parametrize("kind", ["grid_shuffled", "odd_starts"])
def test_box_lists(tm, nbox, kind):
    x, r = w3_small(128, rows=700, cols=520)
    xd = to_dev(x)
    m = dev_map(tm, xd, r)
    rng = np.random.default_rng(nbox)
    if kind == "grid_shuffled":
        starts = [m_ for m_ in (oracle.Map(x, 2, r["dims"], r["strides"], r["box"], 128)
                                .box_start(b) for b in range(m.num_boxes))]
        coords = [starts[i] for i in rng.permutation(len(starts))[:nbox]]
    else:  # x starts 3 elements off the 16-byte grid, first box partly before the tensor
        coords = [[-3 + 64 * (k % 9), 128 * (k // 9) - (5 if k == 0 else 0)] for k in range(nbox)]
    imgs = empty_images(nbox, m.box_bytes)
    tm.tiled_copy(m, coords, imgs)
    check(tm)
    want = oracle.tiled_copy(host_map(x, r), coords=coords)
    np.testing.assert_array_equal(to_host(imgs), want)
    # write the images back through the list into a sentinel tensor (boxes do not overlap)
    dst = full_like(xd, 0x44)
    md = dev_map(tm, dst, r)
    tm.tiled_roundtrip(md, coords, imgs)
    check(tm)
    host_dst = np.full(xd.numel(), 0x44, np.uint8)
    oracle.tiled_roundtrip(host_map(host_dst, r), want, coords=coords)
    np.testing.assert_array_equal(to_host(dst), host_dst)


def test_wholly_outside_box_is_zero(tm):
    x, r = w3_small(128, rows=300, cols=200)
    m = dev_map(tm, to_dev(x), r)
    coords = [[-64, 0], [256, 0], [0, 300], [0, -128]]
    imgs = empty_images(4, m.box_bytes, 0xFF)
    tm.tiled_copy(m, coords, imgs)
    check(tm)
    assert int(imgs.count_nonzero()) == 0


# ---- W4 (reduced): padded rank-3 tensor, ragged boxes, sentinel padding, rank-5 fallback view ----
W4_SMALL = dict(batch=16, rows=70, cols=1000, pitch=1024)


@pytest.mark.parametrize("variant", ["r3_128B", "r3_64B", "r5_none", "r5_128B"])
def test_w4_ragged_and_fallback(tm, variant):
    x = workloads.w4_tensor(**W4_SMALL, seed=41)
    if variant == "r3_128B":
        r = workloads.w4_rank3_map(64, span=128, **W4_SMALL)
    elif variant == "r3_64B":
        r = workloads.w4_rank3_map(32, span=64, **W4_SMALL)
    else:
        r = workloads.w4_rank5_map(**W4_SMALL, span=0 if variant == "r5_none" else 128)
    xd = to_dev(x)
    m = dev_map(tm, xd, r)
    assert m.path == (tm.TM_PATH_FALLBACK if variant.startswith("r5") else tm.TM_PATH_TMA)
    imgs = empty_images(m.num_boxes, m.box_bytes)
    tm.tiled_copy(m, None, imgs)
    check(tm)
    want = oracle.tiled_copy(host_map(x, r), threads=8)
    np.testing.assert_array_equal(to_host(imgs), want)
    # round trip into an all-sentinel tensor: the in-bounds elements come back, padding survives
    dst = torch.from_numpy(np.full(x.size, workloads.SENTINEL_U16, np.uint16).view(np.uint8)).cuda()
    md = dev_map(tm, dst, r)
    tm.tiled_roundtrip(md, None, imgs)
    check(tm)
    assert torch.equal(dst, xd)


# Tensor-map path at ranks 3-5, sizes that give every CTA several box groups: fp32 maps whose
# strides carry padding between dims (all multiples of 16 bytes, so TMA takes them), ragged along
# every dim.  Copy, round trip into a sentinel tensor (padding and the gaps between dims keep their
# bytes), and reduce-add, each against the oracle.
def _high_rank(dims, box, pads):
    strides, st = [], dims[0] * 4
    for i in range(1, len(dims)):
        st += pads[i - 1]
        strides.append(st)
        st *= dims[i]
    return dict(dims=dims, strides=strides, box=box, esize=4), st


HIGH_RANK = {
    "r3": _high_rank([100, 3000, 21], [32, 16, 3], [16, 32]),
    "r4": _high_rank([100, 33, 17, 50], [32, 8, 4, 2], [16, 64, 16]),
    "r5": _high_rank([200, 9, 13, 11, 40], [32, 2, 2, 2, 2], [16, 32, 48, 16]),
}


@pytest.mark.parametrize("case", sorted(HIGH_RANK))
@pytest.mark.parametrize("span", [0, 128])
def test_high_rank_tensor_maps(tm, case, span):
    recipe, nbytes = HIGH_RANK[case]
    r = dict(recipe, span=span)
    d, src = workloads.w5a_tensors(1, nbytes // 4, seed_dst=200 + len(r["dims"]),
                                   seed_src=210 + len(r["dims"]))
    xd = to_dev(d)
    m = dev_map(tm, xd, r)
    assert m.path == tm.TM_PATH_TMA and m.num_boxes > 2000
    imgs = empty_images(m.num_boxes, m.box_bytes)
    tm.tiled_copy(m, None, imgs)
    check(tm)
    want = oracle.tiled_copy(host_map(d, r), threads=8)
    np.testing.assert_array_equal(to_host(imgs), want)
    dst = full_like(xd, 0xC3)
    tm.tiled_roundtrip(dev_map(tm, dst, r), None, imgs)
    check(tm)
    host_dst = np.full(nbytes, 0xC3, np.uint8)
    oracle.tiled_roundtrip(host_map(host_dst, r), want, threads=8)
    np.testing.assert_array_equal(to_host(dst), host_dst)
    sd = to_dev(src)
    tm.tile_reduce_add(m, dev_map(tm, sd, r))
    check(tm)
    hd = d.copy()
    oracle.tile_reduce_add(host_map(hd, r), host_map(src, r), threads=8)
    np.testing.assert_array_equal(to_host(xd), hd.reshape(-1).view(np.uint8))


@pytest.mark.parametrize("case", sorted(HIGH_RANK))
@pytest.mark.parametrize("op", ["add", "max"])
def test_high_rank_vector_reduce(tm, case, op):
    """The vector path's reduce over the same rank 3-5 maps (forced off the tensor reduce): its
    rows are walked with counters over the outer dims stepped with carries."""
    recipe, nbytes = HIGH_RANK[case]
    r = dict(recipe, span=128)
    d, src = workloads.w5a_tensors(1, nbytes // 4, seed_dst=220 + len(r["dims"]),
                                   seed_src=230 + len(r["dims"]))
    dd, sd = to_dev(d), to_dev(src)
    md, ms = dev_map(tm, dd, r), dev_map(tm, sd, r)
    tm.tmap_force_fallback(md)
    code = tm.TM_RED_ADD if op == "add" else tm.TM_RED_MAX
    tm.tile_reduce(md, ms, code)
    check(tm)
    hd = d.copy()
    oracle.tile_reduce(host_map(hd, r), host_map(src, r), oracle.F32,
                       oracle.ADD if op == "add" else oracle.MAX)
    np.testing.assert_array_equal(to_host(dd), hd.reshape(-1).view(np.uint8))


# The vector path's two forms on the same maps: per-window staging and per-thread image loads
# (TM_FB_SEG=0) and segments (TM_FB_SEG=1: contiguous runs of tensor rows or image rows moved by
# bulk copies, realigned by consumer warps).  Ragged boxes along every dim, NaN fill, a base 2
# bytes off alignment, rows of one and of several segments; copy and store directions.
SEG_CASES = {
    # the W4 rank-5 view (dims 0 and 1 contiguous: 2000-byte segments), ragged along dim 2
    "w4r5": (workloads.w4_rank5_map(**W4_SMALL, span=128), 0, False),
    # the same view, box 4 rows along dim 1 (the last box of a group holds 2 rows), NaN fill
    "w4r5_dim1_ragged": (dict(workloads.w4_rank5_map(**W4_SMALL, span=128), box=[64, 4, 16, 1, 1],
                              nan=True), 0, True),
    # one-row segments: rows of 1000 elements at a 2048-byte pitch, the base 2 bytes off
    "rows_offset": (dict(dims=[1000, 70, 16], strides=[2048, 70 * 2048], box=[64, 32, 2],
                         span=128, esize=2), 2, False),
    # dims 0 and 1 contiguous, unswizzled 48-byte image rows, 3 boxes along dim 0
    "fused_48B": (dict(dims=[60, 9, 70, 16], strides=[120, 1080, 70 * 2048], box=[24, 3, 8, 1],
                       span=0, esize=2), 0, False),
}


@pytest.mark.parametrize("case", sorted(SEG_CASES))
@pytest.mark.parametrize("seg", ["0", "1"])
def test_vector_copy_forms(tm, monkeypatch, case, seg):
    monkeypatch.setenv("TM_FB_SEG", seg)
    r, offset, nan = SEG_CASES[case]
    x = workloads.w4_tensor(**W4_SMALL, seed=43)
    dt = tm.TM_BF16 if nan else None
    xd = to_dev(x)
    m = dev_map(tm, xd, r, offset=offset, dtype=dt)
    assert m.path == tm.TM_PATH_FALLBACK
    imgs = empty_images(m.num_boxes, m.box_bytes)
    tm.tiled_copy(m, None, imgs)
    check(tm)
    want = oracle.tiled_copy(host_map(x, r, offset=offset, dtype=dt), threads=8)
    if nan:
        assert_nan_fill(to_host(imgs), want, dt, tm)
    else:
        np.testing.assert_array_equal(to_host(imgs), want)
    # store direction: the oracle's images back into a sentinel-filled tensor (only in-bounds
    # elements are written; padding and everything outside the map keep the sentinel)
    hin = torch.from_numpy(want.copy()).cuda()
    dst = full_like(xd, 0xA5)
    tm.tiled_roundtrip(dev_map(tm, dst, r, offset=offset, dtype=dt), None, hin)
    check(tm)
    hdst = np.full(xd.numel(), 0xA5, np.uint8)
    oracle.tiled_roundtrip(host_map(hdst, r, offset=offset, dtype=dt), want)
    np.testing.assert_array_equal(to_host(dst), hdst)


# ---- W5a (reduced): fp32 reduce-add, [Book-TMA] §"TMA reduce，把“搬运”和“归约”合并" ----------------
@pytest.mark.parametrize("span", [128, 0])
@pytest.mark.parametrize("force_fallback", [False, True])
def test_w5a_reduce_add(tm, span, force_fallback):
    d, s = workloads.w5a_tensors(rows=300, cols=200, seed_dst=7, seed_src=8)
    r = workloads.w5a_map(rows=300, cols=200, span=span)
    dd, sd = to_dev(d), to_dev(s)
    md, ms = dev_map(tm, dd, r), dev_map(tm, sd, r)
    if force_fallback:
        tm.tmap_force_fallback(md)
    tm.tile_reduce_add(md, ms)
    check(tm)
    hd = d.copy()
    oracle.tile_reduce_add(host_map(hd, r), host_map(s, r))
    np.testing.assert_array_equal(to_host(dd).view(np.uint32), hd.reshape(-1).view(np.uint32))


# ---- W5b (reduced): the ring, [MLSys-TMA] §"把 TMA 放进 pipeline" ---------------------------------
@pytest.mark.parametrize("span", [128, 0])
@pytest.mark.parametrize("stages", [2, 4, 6])
def test_w5b_ring_checksums(tm, span, stages):
    a, b = workloads.w5b_tensors(m=380, k=248, n=376, seed_a=9, seed_b=10)
    ra, rb = workloads.w5b_maps(m=380, k=248, n=376, span=span)
    ad, bd = to_dev(a), to_dev(b)
    ma, mb = dev_map(tm, ad, ra), dev_map(tm, bd, rb)
    n = ma.num_boxes
    assert n == mb.num_boxes == 12
    cs_a = guarded(4 * n, 0).view(torch.float32)
    cs_b = guarded(4 * n, 0).view(torch.float32)
    bits_a = guarded(8 * n, 0).view(torch.int64)
    bits_b = guarded(8 * n, 0).view(torch.int64)
    tm.stream_tiles(ma, mb, stages, cs_a, cs_b, bits_a, bits_b)
    check(tm)
    wa, wb, wba, wbb = oracle.stream_checksums(host_map(a, ra), host_map(b, rb))
    np.testing.assert_array_equal(to_host(cs_a).view(np.uint32), wa.view(np.uint32))
    np.testing.assert_array_equal(to_host(cs_b).view(np.uint32), wb.view(np.uint32))
    np.testing.assert_array_equal(to_host(bits_a).astype(np.uint64), wba)
    np.testing.assert_array_equal(to_host(bits_b).astype(np.uint64), wbb)


@pytest.mark.parametrize("stages", [2, 4])
def test_w5b_ring_checksums_special_values(tm, stages):
    """Tiles of arbitrary bf16 patterns (every special pair, their neighbours and uniform random
    bits: subnormals, infinities, NaNs): the fp32 row sums bit for bit against the oracle where
    they are numbers and NaN where the oracle's are (the payload of an operation's NaN is open);
    the sums of the 16-bit patterns exactly."""
    a0, b0 = workloads.w5b_tensors(m=380, k=248, n=376, seed_a=9, seed_b=10)
    finite = [0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x807F, 0x0080, 0x8080, 0x3F80, 0xBF80]

    def mix(x0, seed, which):
        # finite special patterns everywhere; the full mix (NaNs, infinities, the largest
        # finite) in the first 64 rows only, so that some tiles sum to numbers and some do not
        sp = workloads.special_reduce_operands("bf16", *x0.shape, seed=seed)[which].reshape(x0.shape)
        x = x0.copy()
        pick = np.isin(sp, finite)
        x[pick] = sp[pick]
        x[:64] = sp[:64]
        return x

    a, b = mix(a0, 31, 0), mix(b0, 32, 1)
    ra, rb = workloads.w5b_maps(m=380, k=248, n=376, span=128)
    ad, bd = to_dev(a), to_dev(b)
    ma, mb = dev_map(tm, ad, ra), dev_map(tm, bd, rb)
    n = ma.num_boxes
    cs_a = guarded(4 * n, 0).view(torch.float32)
    cs_b = guarded(4 * n, 0).view(torch.float32)
    bits_a = guarded(8 * n, 0).view(torch.int64)
    bits_b = guarded(8 * n, 0).view(torch.int64)
    tm.stream_tiles(ma, mb, stages, cs_a, cs_b, bits_a, bits_b)
    check(tm)
    wa, wb, wba, wbb = oracle.stream_checksums(host_map(a, ra), host_map(b, rb))
    for got, want in ((to_host(cs_a).view(np.float32), wa), (to_host(cs_b).view(np.float32), wb)):
        nan = np.isnan(want)
        assert nan.any() and not nan.all()  # the tiles exercise both outcomes
        np.testing.assert_array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))
        assert np.isnan(got[nan]).all()
    np.testing.assert_array_equal(to_host(bits_a).astype(np.uint64), wba)
    np.testing.assert_array_equal(to_host(bits_b).astype(np.uint64), wbb)


# Many laps of the ring on every CTA: tiles of every supported height, ragged in both dims (296
# columns = 4 full 64-column boxes + 40; rows not a multiple of the tile), with one consumer group,
# two (even and odd tiles), and the row-pairs read order (the ungrouped bank-conflict control,
# whose results must not change), and with the tile loads' L2 evict-first policy dropped (a cache
# policy cannot change the bytes read).  A and B are both M x 296, different seeds.
RING_LAPS_ROWS = {32: 32000 - 5, 64: 48000 - 7, 128: 32000 - 9, 256: 64000 - 11}


@pytest.mark.parametrize("rows", [32, 64, 128, 256])
@pytest.mark.parametrize("mode", ["two_groups", "one_group", "row_pairs", "no_evict_first"])
def test_w5b_ring_many_laps(tm, monkeypatch, rows, mode):
    stages = 3 if rows == 256 else 4
    monkeypatch.setenv("TM_RING_GROUPS", "1" if mode == "one_group" else "2")
    monkeypatch.setenv("TM_RING_ROW_PAIRS", "1" if mode == "row_pairs" else "0")
    monkeypatch.setenv("TM_RING_EVICT_FIRST", "0" if mode == "no_evict_first" else "1")
    m = RING_LAPS_ROWS[rows]
    a = workloads.normal_bf16((m, 296), 60 + rows)
    b = workloads.normal_bf16((m, 296), 61 + rows)
    r = dict(dims=[296, m], strides=[592], box=[64, rows], span=128, esize=2)
    ad, bd = to_dev(a), to_dev(b)
    ma, mb = dev_map(tm, ad, r), dev_map(tm, bd, r)
    n = ma.num_boxes
    assert n == 5 * -(-m // rows) and n > 1000
    cs_a = guarded(4 * n, 0).view(torch.float32)
    cs_b = guarded(4 * n, 0).view(torch.float32)
    bits_a = guarded(8 * n, 0).view(torch.int64)
    bits_b = guarded(8 * n, 0).view(torch.int64)
    tm.stream_tiles(ma, mb, stages, cs_a, cs_b, bits_a, bits_b)
    check(tm)
    wa, wb, wba, wbb = oracle.stream_checksums(host_map(a, r), host_map(b, r),
                                               threads=oracle.host_cores())
    np.testing.assert_array_equal(to_host(cs_a).view(np.uint32), wa.view(np.uint32))
    np.testing.assert_array_equal(to_host(cs_b).view(np.uint32), wb.view(np.uint32))
    np.testing.assert_array_equal(to_host(bits_a).astype(np.uint64), wba)
    np.testing.assert_array_equal(to_host(bits_b).astype(np.uint64), wbb)


# ---- brute force: random tiny maps of every rank, swizzle and element size ----------------------
def random_recipe(rng, span, aligned):
    rank = int(rng.integers(1, 6))
    es = int(rng.choice([2, 4])) if span else int(rng.choice([1, 2, 4, 8]))
    box = [int(rng.integers(1, 5)) for _ in range(rank)]
    box[0] = span // es if span else (16 // es) * int(rng.integers(1, 3))
    dims = [int(rng.integers(1, 6)) for _ in range(rank)]
    dims[0] = int(rng.integers(1, box[0] + 7))
    strides, step = [], dims[0] * es
    order = rng.permutation(np.arange(1, rank))
    st = [0] * rank
    for dd in order:
        pad = int(rng.integers(0, 3)) * es
        if aligned:
            step = (step + 15) // 16 * 16
        st[dd] = step
        step = step * dims[dd] + pad
    strides = [st[i] for i in range(1, rank)]
    return dict(dims=dims, strides=strides, box=box, span=span, esize=es), step + 64


@pytest.mark.parametrize("span", [0, 32, 64, 128])
@pytest.mark.parametrize("aligned", [True, False])
@pytest.mark.parametrize("seg", ["auto", "forced"])
def test_brute_force_tiny(tm, monkeypatch, span, aligned, seg):
    if seg == "forced":  # the vector copy's segment form whenever the layout allows it
        monkeypatch.setenv("TM_FB_SEG", "1")
    rng = np.random.default_rng(500 + span + aligned)
    for _ in range(25):
        r, nbytes = random_recipe(rng, span, aligned)
        x = rng.integers(0, 256, size=nbytes, dtype=np.uint16).astype(np.uint8)
        xd = to_dev(x)
        m = dev_map(tm, xd, r)
        coords = [[int(rng.integers(-3, d + 4)) for d in r["dims"]] for _ in range(3)]
        coords.append([0] * len(r["dims"]))
        imgs = empty_images(len(coords), m.box_bytes)
        tm.tiled_copy(m, coords, imgs)
        check(tm)
        want = oracle.tiled_copy(host_map(x, r), coords=coords)
        np.testing.assert_array_equal(to_host(imgs), want, err_msg=f"{r} {coords} path={m.path}")
        # whole grid, then back into a sentinel copy
        g = empty_images(m.num_boxes, m.box_bytes)
        tm.tiled_copy(m, None, g)
        dst = full_like(xd, 0xC3)
        md = dev_map(tm, dst, r)
        tm.tiled_roundtrip(md, None, g)
        check(tm)
        hg = oracle.tiled_copy(host_map(x, r))
        np.testing.assert_array_equal(to_host(g), hg)
        hdst = np.full_like(x, 0xC3)
        oracle.tiled_roundtrip(host_map(hdst, r), hg)
        np.testing.assert_array_equal(to_host(dst), hdst, err_msg=f"{r} store path={md.path}")


def test_store_keeps_padding_after_a_ragged_row_end(tm):
    """Rows whose in-bounds part ends inside a 16-byte unit: the bytes after it stay untouched
    (the tensor store would write the whole unit, so these maps store on the vector path)."""
    for es in (2, 4):
        for d0 in range(1, 9):
            r = dict(dims=[d0, 3], strides=[32], box=[16 // es, 2], span=0, esize=es)
            x = (np.arange(160) % 251 + 1).astype(np.uint8)
            xd = to_dev(x)
            m = dev_map(tm, xd, r)
            g = empty_images(m.num_boxes, m.box_bytes)
            tm.tiled_copy(m, None, g)
            dst = full_like(xd, 0xC3)
            tm.tiled_roundtrip(dev_map(tm, dst, r), None, g)
            check(tm)
            hdst = np.full_like(x, 0xC3)
            oracle.tiled_roundtrip(host_map(hdst, r), oracle.tiled_copy(host_map(x, r)))
            np.testing.assert_array_equal(to_host(dst), hdst, err_msg=f"esize {es} dim0 {d0}")


def test_reduce_add_ragged_row_end(tm):
    d, s = workloads.w5a_tensors(rows=40, cols=35, seed_dst=11, seed_src=12)
    pad = np.full((40, 40), np.float32(-0.0), np.float32)  # 160-byte rows, 140 in bounds
    pad[:, :35] = d
    r = dict(dims=[35, 40], strides=[160], box=[32, 16], span=128, esize=4)
    spad = np.zeros((40, 40), np.float32)
    spad[:, :35] = s
    dd, sd = to_dev(pad), to_dev(spad)
    tm.tile_reduce_add(dev_map(tm, dd, r), dev_map(tm, sd, r))
    check(tm)
    hd = pad.copy()
    oracle.tile_reduce_add(host_map(hd, r), host_map(spad, r))
    np.testing.assert_array_equal(to_host(dd).view(np.uint32), hd.reshape(-1).view(np.uint32))


@pytest.mark.parametrize("force_fallback", [False, True])
def test_big_boxes_single_stage(tm, force_fallback):
    """128 KiB boxes: one stage per CTA on the tensor-map path, one image stage on the vector path."""
    x = workloads.normal_bf16((9, 300, 64), 21)
    r = dict(dims=[64, 300, 9], strides=[128, 300 * 128], box=[64, 256, 4], span=128, esize=2)
    xd = to_dev(x)
    m = dev_map(tm, xd, r)
    if force_fallback:
        tm.tmap_force_fallback(m)
    assert (m.num_boxes, m.box_bytes) == (6, 131072)
    imgs = empty_images(m.num_boxes, m.box_bytes)
    tm.tiled_copy(m, None, imgs)
    check(tm)
    want = oracle.tiled_copy(host_map(x, r))
    np.testing.assert_array_equal(to_host(imgs), want)
    dst = full_like(xd, 0x66)
    md = dev_map(tm, dst, r)
    if force_fallback:
        tm.tmap_force_fallback(md)
    tm.tiled_roundtrip(md, None, imgs)
    check(tm)
    assert torch.equal(dst, xd)
    d, s = workloads.w5a_tensors(rows=520, cols=32, seed_dst=13, seed_src=14)
    rr = dict(dims=[32, 520], strides=[128], box=[32, 256], span=128, esize=4)
    dd, sd = to_dev(d), to_dev(s)
    mdd = dev_map(tm, dd, rr)
    if force_fallback:
        tm.tmap_force_fallback(mdd)
    tm.tile_reduce_add(mdd, dev_map(tm, sd, rr))
    check(tm)
    hd = d.copy()
    oracle.tile_reduce_add(host_map(hd, rr), host_map(s, rr))
    np.testing.assert_array_equal(to_host(dd).view(np.uint32), hd.reshape(-1).view(np.uint32))


def test_guard_bands_catch_a_stray_byte():
    """The guard check that runs after every GPU test sees a byte written just past a buffer (and
    just before one).  The stray bytes are written by torch into the guard band itself, which is
    allocated memory, so nothing here accesses memory out of bounds."""
    import gpu_util
    for where in ("after", "before"):
        body = gpu_util.guarded(64, 0)
        buf = gpu_util._guarded[-1][0]
        buf[gpu_util.GUARD + 64 if where == "after" else gpu_util.GUARD - 1] = 1
        with pytest.raises(AssertionError):
            gpu_util.check_guards()
        assert not gpu_util._guarded and int(body.sum()) == 0


# ---- bounded waits: a wait that nothing completes gives up and reports, the GPU stays usable -----
def test_wait_timeout_is_reported_and_recoverable(tm):
    tm.tm_selftest_wait_timeout(50_000_000)
    rc = tm.tm_stream_check()
    assert rc == tm.TM_ETIMEOUT
    assert "self-test" in tm.tm_last_error()
    assert tm.tm_stream_check() == tm.TM_OK  # the status word was cleared
    x, r = w3_small(128, rows=256, cols=128)
    m = dev_map(tm, to_dev(x), r)
    imgs = empty_images(m.num_boxes, m.box_bytes)
    tm.tiled_copy(m, None, imgs)
    check(tm)
    np.testing.assert_array_equal(to_host(imgs), oracle.tiled_copy(host_map(x, r)))
