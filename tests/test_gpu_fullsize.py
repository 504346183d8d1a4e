"""Parity at the workloads' full sizes, in the launch configuration the benchmark times (library
defaults).  The oracle computes sampled outputs (whole boxes or tiles, one by one); properties
that hold at any size cover the rest: a round trip restores the tensor exactly, padding
sentinels survive, and the ring's checksums are compared for every tile.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_util import dev_map, full_like, guarded, host_map, to_dev, to_host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tm():
    import async_bulk_tensor_tmap_gb300 as m  # raises if the CUDA library is missing
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def check(tm):
    torch.cuda.synchronize()
    assert tm.tm_stream_check() == tm.TM_OK, tm.tm_last_error()


def sample_boxes(n, k, seed):
    rng = np.random.default_rng(seed)
    picks = set(rng.choice(n, size=min(k, n), replace=False).tolist())
    return sorted(picks | {0, n - 1})


def assert_sampled_images(imgs_dev, om, boxes):
    bb = om.box_bytes
    got = to_host(imgs_dev)
    for b in boxes:
        want = oracle.image(om, om.box_start(b))
        np.testing.assert_array_equal(got[b * bb:(b + 1) * bb], want, err_msg=f"box {b}")


def test_w3_full_copy_and_roundtrip(tm):
    x = workloads.w3_tensor()
    r = workloads.w3_map()
    xd = to_dev(x)
    m = dev_map(tm, xd, r)
    imgs = torch.empty(m.num_boxes * m.box_bytes, dtype=torch.uint8, device="cuda")
    tm.tiled_copy(m, None, imgs)
    check(tm)
    assert_sampled_images(imgs, host_map(x, r), sample_boxes(m.num_boxes, 64, 3))
    dst = full_like(xd, 0x5C)
    tm.tiled_roundtrip(dev_map(tm, dst, r), None, imgs)
    check(tm)
    assert torch.equal(dst, xd)


@pytest.mark.parametrize("variant", ["r3_128B", "r3_64B", "r5_128B"])
def test_w4_full_copy_and_roundtrip(tm, variant):
    x = workloads.w4_tensor()
    if variant == "r3_128B":
        r = workloads.w4_rank3_map(64, span=128)
    elif variant == "r3_64B":
        r = workloads.w4_rank3_map(32, span=64)
    else:
        r = workloads.w4_rank5_map(span=128)
    xd = to_dev(x)
    m = dev_map(tm, xd, r)
    assert m.path == (tm.TM_PATH_FALLBACK if variant.startswith("r5") else tm.TM_PATH_TMA)
    imgs = torch.empty(m.num_boxes * m.box_bytes, dtype=torch.uint8, device="cuda")
    tm.tiled_copy(m, None, imgs)
    check(tm)
    assert_sampled_images(imgs, host_map(x, r), sample_boxes(m.num_boxes, 48, 4))
    sent = np.full(x.size, workloads.SENTINEL_U16, np.uint16)
    dst = torch.from_numpy(sent.view(np.uint8)).cuda()
    tm.tiled_roundtrip(dev_map(tm, dst, r), None, imgs)
    check(tm)
    assert torch.equal(dst, xd)  # in-bounds elements restored, padding sentinel untouched


def test_w5a_full_reduce_add(tm):
    d, s = workloads.w5a_tensors()
    r = workloads.w5a_map()
    dd, sd = to_dev(d), to_dev(s)
    tm.tile_reduce_add(dev_map(tm, dd, r), dev_map(tm, sd, r))
    check(tm)
    got = to_host(dd).view(np.float32).reshape(d.shape)
    md, ms = host_map(d, r), host_map(s, r)
    nb0 = -(-r["dims"][0] // r["box"][0])
    rng = np.random.default_rng(5)
    starts = [0, md.num_boxes - 8] + rng.integers(0, md.num_boxes - 8, size=14).tolist()
    for b0 in starts:
        oracle.tile_reduce_add(md, ms, b0=b0, b1=b0 + 8)  # updates the host dst in place
        for b in range(b0, b0 + 8):
            k0, k1 = b % nb0, b // nb0
            rows = slice(k1 * 128, k1 * 128 + 128)
            cols = slice(k0 * 32, k0 * 32 + 32)
            np.testing.assert_array_equal(got[rows, cols].view(np.uint32),
                                          d[rows, cols].view(np.uint32), err_msg=f"box {b}")


def test_w5b_full_ring_every_tile(tm):
    a, b = workloads.w5b_tensors()
    ra, rb = workloads.w5b_maps()
    ad, bd = to_dev(a), to_dev(b)
    ma, mb = dev_map(tm, ad, ra), dev_map(tm, bd, rb)
    n = ma.num_boxes
    cs_a = guarded(4 * n, 0).view(torch.float32)
    cs_b = guarded(4 * n, 0).view(torch.float32)
    bits_a = guarded(8 * n, 0).view(torch.int64)
    bits_b = guarded(8 * n, 0).view(torch.int64)
    tm.stream_tiles(ma, mb, 4, cs_a, cs_b, bits_a, bits_b)
    check(tm)
    wa, wb, wba, wbb = oracle.stream_checksums(host_map(a, ra), host_map(b, rb),
                                               threads=oracle.host_cores())
    np.testing.assert_array_equal(to_host(cs_a).view(np.uint32), wa.view(np.uint32))
    np.testing.assert_array_equal(to_host(cs_b).view(np.uint32), wb.view(np.uint32))
    np.testing.assert_array_equal(to_host(bits_a).astype(np.uint64), wba)
    np.testing.assert_array_equal(to_host(bits_b).astype(np.uint64), wbb)
