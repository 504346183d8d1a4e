"""Parity at the workloads' full sizes, in the launch configuration the benchmark times (library
defaults).  Every output is compared with the oracle, computed on all host cores: every image of
W3 and of the three W4 maps, the whole W5a destination after the reduce-add, and every ring tile's
checksums; the round trips must also restore the tensor exactly with its padding sentinels.
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


def assert_all_images(imgs_dev, om):
    """Every image the GPU wrote equals the oracle's; a mismatch names its first box."""
    got = to_host(imgs_dev)
    want = oracle.tiled_copy(om, threads=oracle.host_cores())
    if not np.array_equal(got, want):
        bad = int(np.flatnonzero(got != want)[0]) // om.box_bytes
        raise AssertionError(f"image of box {bad} (of {om.num_boxes}) differs from the oracle")


def test_w3_full_copy_and_roundtrip(tm):
    x = workloads.w3_tensor()
    r = workloads.w3_map()
    xd = to_dev(x)
    m = dev_map(tm, xd, r)
    imgs = torch.empty(m.num_boxes * m.box_bytes, dtype=torch.uint8, device="cuda")
    tm.tiled_copy(m, None, imgs)
    check(tm)
    assert_all_images(imgs, host_map(x, r))
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
    assert_all_images(imgs, host_map(x, r))
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
    got = to_host(dd).view(np.uint32).reshape(d.shape)
    md, ms = host_map(d, r), host_map(s, r)
    oracle.tile_reduce_add(md, ms, threads=oracle.host_cores())  # updates the host dst in place
    want = d.view(np.uint32)
    if not np.array_equal(got, want):
        row, col = (int(v[0]) for v in np.nonzero(got != want))
        raise AssertionError(f"dst[{row}, {col}] differs from the oracle "
                             f"(box {(row // 128) * (-(-r['dims'][0] // 32)) + col // 32})")


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
