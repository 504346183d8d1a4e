"""The streaming kernels' dynamic work split: a launch takes its items from a counter of its
stream (zero at launch, set back to zero by the launch's last CTA), so faster CTAs take more
items.  What must hold: every item is done exactly once, on any number of streams at once and over
any number of launches in a row; a launch captured into a CUDA graph (static split) replays
correctly; the static split (TM_DYNAMIC=0) gives the same bytes.  The fp32 reduce-add is the
sharpest check: an item lost or done twice changes the destination.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import dev_map, host_map, to_dev, to_host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tm():
    import async_bulk_tensor_tmap_gb300 as m  # raises if the CUDA library is missing
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def reduce_case(rows, cols, seed):
    d, s = workloads.w5a_tensors(rows, cols, seed_dst=seed, seed_src=seed + 1)
    return d, s, workloads.w5a_map(rows, cols)


def oracle_sum(d, s, r, times):
    want = d.copy()
    md, ms = host_map(want, r), host_map(s, r)
    for _ in range(times):
        oracle.tile_reduce_add(md, ms, threads=oracle.host_cores())
    return want


def test_reduce_add_on_four_streams_at_once(tm):
    """Four streams, each with its own tensors, three reduce-adds each, all in flight together."""
    cases = [reduce_case(1536 + 128 * i, 1024, 60 + 2 * i) for i in range(4)]
    streams = [torch.cuda.Stream() for _ in cases]
    devs = []
    for d, s, r in cases:
        dd, sd = to_dev(d), to_dev(s)
        devs.append((dd, sd, dev_map(tm, dd, r), dev_map(tm, sd, r)))
    torch.cuda.synchronize()
    for _ in range(3):
        for st, (dd, sd, md, ms) in zip(streams, devs):
            tm.tile_reduce_add(md, ms, st)
    torch.cuda.synchronize()
    assert tm.tm_stream_check() == tm.TM_OK, tm.tm_last_error()
    for (d, s, r), (dd, _, _, _) in zip(cases, devs):
        got = to_host(dd).view(np.uint32)
        np.testing.assert_array_equal(got, oracle_sum(d, s, r, 3).reshape(-1).view(np.uint32))


def test_many_launches_in_a_row_on_one_stream(tm):
    """Twelve copies back to back on one stream (the counter must be back at zero after each)."""
    x = workloads.w3_tensor(1000, 776, seed=70)
    r = workloads.w3_map(1000, 776)
    xd = to_dev(x)
    m = dev_map(tm, xd, r)
    want = oracle.tiled_copy(host_map(x, r), threads=oracle.host_cores())
    outs = [torch.empty(m.num_boxes * m.box_bytes, dtype=torch.uint8, device="cuda") for _ in range(12)]
    for o in outs:
        tm.tiled_copy(m, None, o)
    torch.cuda.synchronize()
    assert tm.tm_stream_check() == tm.TM_OK, tm.tm_last_error()
    for o in outs:
        assert np.array_equal(to_host(o), want)


def test_captured_launch_replays(tm):
    """A reduce-add captured into a CUDA graph (static split under capture), replayed twice,
    beside a direct launch on another stream."""
    d, s, r = reduce_case(1024, 1536, 80)
    d2, s2, r2 = reduce_case(768, 1024, 82)
    dd, sd = to_dev(d), to_dev(s)
    dd2, sd2 = to_dev(d2), to_dev(s2)
    md, ms = dev_map(tm, dd, r), dev_map(tm, sd, r)
    md2, ms2 = dev_map(tm, dd2, r2), dev_map(tm, sd2, r2)
    cap = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=cap):
        tm.tile_reduce_add(md, ms, cap)
    other = torch.cuda.Stream()
    g.replay()
    tm.tile_reduce_add(md2, ms2, other)
    g.replay()
    torch.cuda.synchronize()
    assert tm.tm_stream_check() == tm.TM_OK, tm.tm_last_error()
    np.testing.assert_array_equal(to_host(dd).view(np.uint32),
                                  oracle_sum(d, s, r, 2).reshape(-1).view(np.uint32))
    np.testing.assert_array_equal(to_host(dd2).view(np.uint32),
                                  oracle_sum(d2, s2, r2, 1).reshape(-1).view(np.uint32))


@pytest.mark.parametrize("dynamic", ["0", "1"])
def test_static_and_dynamic_split_agree(tm, monkeypatch, dynamic):
    """Copy, round trip and reduce-add of ragged shapes with either split."""
    monkeypatch.setenv("TM_DYNAMIC", dynamic)
    x = workloads.w3_tensor(1000, 776, seed=71)
    r = workloads.w3_map(1000, 776)
    xd = to_dev(x)
    m = dev_map(tm, xd, r)
    imgs = torch.empty(m.num_boxes * m.box_bytes, dtype=torch.uint8, device="cuda")
    tm.tiled_copy(m, None, imgs)
    back = torch.zeros_like(xd)
    tm.tiled_roundtrip(dev_map(tm, back, r), None, imgs)
    d, s, rr = reduce_case(700, 424, 90)
    dd, sd = to_dev(d), to_dev(s)
    tm.tile_reduce_add(dev_map(tm, dd, rr), dev_map(tm, sd, rr))
    torch.cuda.synchronize()
    assert tm.tm_stream_check() == tm.TM_OK, tm.tm_last_error()
    assert np.array_equal(to_host(imgs), oracle.tiled_copy(host_map(x, r)))
    assert torch.equal(back, xd)
    np.testing.assert_array_equal(to_host(dd).view(np.uint32),
                                  oracle_sum(d, s, rr, 1).reshape(-1).view(np.uint32))


def test_vector_path_segments_on_three_streams_and_in_a_row(tm):
    """The vector path's segment kernels (the W4 rank-5 view, a 200-byte stride) take their items
    the same way: copies and round trips on three streams at once, twice each, then four copies in
    a row on one stream; every image and every restored tensor against the oracle."""
    kw = dict(batch=16, rows=70, cols=1000, pitch=1024)
    x = workloads.w4_tensor(**kw, seed=73)
    r = workloads.w4_rank5_map(**kw, span=128)
    xd = to_dev(x)
    m = dev_map(tm, xd, r)
    assert m.path == tm.TM_PATH_FALLBACK
    want = oracle.tiled_copy(host_map(x, r), threads=oracle.host_cores())
    sent = np.full(x.size, workloads.SENTINEL_U16, np.uint16)
    streams = [torch.cuda.Stream() for _ in range(3)]
    imgs = [torch.empty(m.num_boxes * m.box_bytes, dtype=torch.uint8, device="cuda") for _ in streams]
    backs = [torch.from_numpy(sent.view(np.uint8).copy()).cuda() for _ in streams]
    bmaps = [dev_map(tm, bk, r) for bk in backs]
    torch.cuda.synchronize()
    for _ in range(2):
        for st, im, bm in zip(streams, imgs, bmaps):
            tm.tiled_copy(m, None, im, st)
            tm.tiled_roundtrip(bm, None, im, st)
    torch.cuda.synchronize()
    assert tm.tm_stream_check() == tm.TM_OK, tm.tm_last_error()
    for im, bk in zip(imgs, backs):
        assert np.array_equal(to_host(im), want)
        assert torch.equal(bk, xd)
    outs = [torch.empty_like(imgs[0]) for _ in range(4)]
    for o in outs:
        tm.tiled_copy(m, None, o)
    torch.cuda.synchronize()
    assert tm.tm_stream_check() == tm.TM_OK, tm.tm_last_error()
    for o in outs:
        assert np.array_equal(to_host(o), want)
