"""tiled_copy_noalloc: the tiled copy for callers that must not allocate device memory (code that
runs while another allocator owns all device memory, under a hard memory cap, or in loops that
cannot afford an allocator call).  Its scratch is a fixed array inside the library, so its output
must equal that of the allocating tiled_copy on the same inputs -- on two calls in a row, the
second seeing whatever the first left in the shared scratch.

Named to be collected last, so that a run stopping at the first failure has run everything else.
Runs the same alone in a fresh process and after the other tests.
"""
import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tm():
    import async_bulk_tensor_tmap_gb300 as m  # raises if the CUDA library is missing
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


def _map(tm, buf, rows, cols):
    r = workloads.w3_map(rows, cols)
    m = tm.tmap_encode(tm.TM_BF16, buf, r["dims"], r["strides"], r["box"],
                       swizzle=tm.TM_SWIZZLE_128B)
    return m


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x).reshape(-1).view(np.uint8).copy()).cuda()


def test_noalloc_matches_tiled_copy_on_two_calls(tm):
    x = workloads.w3_tensor(700, 520, seed=77)
    xd = _dev(x)
    m = _map(tm, xd, 700, 520)
    rng = np.random.default_rng(3)
    starts = []
    for b in range(m.num_boxes):
        k0, k1 = b % m.d.nbox[0], b // m.d.nbox[0]
        starts.append([int(k0 * 64), int(k1 * 128)])
    lists = [
        [starts[i] for i in rng.permutation(len(starts))[:37]],            # tensor-map path
        [[-3 + 64 * (k % 9), 128 * (k // 9)] for k in range(23)],          # vector path
    ]
    for coords in lists:
        want = torch.full((len(coords) * m.box_bytes,), 0x11, dtype=torch.uint8, device="cuda")
        tm.tiled_copy(m, coords, want)
        torch.cuda.synchronize()
        assert tm.tm_stream_check() == tm.TM_OK, tm.tm_last_error()
        for _ in range(2):  # two calls in a row share the scratch
            got = torch.full_like(want, 0x22)
            tm.tiled_copy_noalloc(m, coords, got)
            assert torch.equal(got, want)
    # the whole grid (no list) as well
    want = torch.zeros(m.num_boxes * m.box_bytes, dtype=torch.uint8, device="cuda")
    tm.tiled_copy(m, None, want)
    torch.cuda.synchronize()
    for _ in range(2):
        got = torch.full_like(want, 0x33)
        tm.tiled_copy_noalloc(m, None, got)
        assert torch.equal(got, want)


def test_noalloc_rejects_lists_beyond_its_scratch(tm):
    x = workloads.w3_tensor(256, 128, seed=5)
    xd = _dev(x)
    m = _map(tm, xd, 256, 128)
    n = tm.TM_NOALLOC_MAX_BOXES + 1
    coords = [[0, 0]] * n
    images = torch.empty(n * m.box_bytes, dtype=torch.uint8, device="cuda")
    with pytest.raises(tm.TmapError) as e:
        tm.tiled_copy_noalloc(m, coords, images)
    assert e.value.code == tm.TM_ERANGE
    assert "at most" in str(e.value)


def test_noalloc_vector_path_whole_grid(tm):
    """A map the tensor-map hardware cannot take (the W4 rank-5 view, 200-byte stride), its whole
    grid: the no-allocation copy gives the allocating copy's images."""
    kw = dict(batch=16, rows=70, cols=1000, pitch=1024)
    x = workloads.w4_tensor(**kw, seed=45)
    r = workloads.w4_rank5_map(**kw, span=128)
    xd = _dev(x)
    m = tm.tmap_encode(tm.TM_BF16, xd, r["dims"], r["strides"], r["box"],
                       swizzle=tm.TM_SWIZZLE_128B)
    assert m.path == tm.TM_PATH_FALLBACK
    want = torch.zeros(m.num_boxes * m.box_bytes, dtype=torch.uint8, device="cuda")
    tm.tiled_copy(m, None, want)
    torch.cuda.synchronize()
    assert tm.tm_stream_check() == tm.TM_OK, tm.tm_last_error()
    for _ in range(2):
        got = torch.full_like(want, 0x44)
        tm.tiled_copy_noalloc(m, None, got)
        assert torch.equal(got, want)


def test_noalloc_small_boxes_share_stages(tm):
    """512-byte boxes (128B swizzle), packed several to a stage in slots on their swizzle period:
    the no-allocation copy gives the allocating copy's images."""
    x = workloads.w3_tensor(300, 392, seed=46)
    xd = _dev(x)
    m = tm.tmap_encode(tm.TM_BF16, xd, [392, 300], [784], [64, 4], swizzle=tm.TM_SWIZZLE_128B)
    assert m.path == tm.TM_PATH_TMA and m.box_bytes == 512
    want = torch.zeros(m.num_boxes * m.box_bytes, dtype=torch.uint8, device="cuda")
    tm.tiled_copy(m, None, want)
    torch.cuda.synchronize()
    assert tm.tm_stream_check() == tm.TM_OK, tm.tm_last_error()
    got = torch.full_like(want, 0x55)
    tm.tiled_copy_noalloc(m, None, got)
    assert torch.equal(got, want)


def test_noalloc_on_a_non_default_stream(tm):
    """The caller's own non-blocking stream: the status word is cleared and the box list uploaded
    on that stream, the copy runs there, and the call reads the status back before returning.
    Images as tiled_copy's, for a listed-box call (list staged in the scratch) and the whole grid."""
    x = workloads.w3_tensor(520, 700, seed=78)
    xd = _dev(x)
    m = _map(tm, xd, 520, 700)
    coords = [[int(64 * (b % m.d.nbox[0])), int(128 * (b // m.d.nbox[0]))]
              for b in np.random.default_rng(9).permutation(m.num_boxes)[:29]]
    s = torch.cuda.Stream()
    for lst in (coords, None):
        n = len(lst) if lst is not None else m.num_boxes
        want = torch.zeros(n * m.box_bytes, dtype=torch.uint8, device="cuda")
        tm.tiled_copy(m, lst, want)
        torch.cuda.synchronize()
        assert tm.tm_stream_check() == tm.TM_OK, tm.tm_last_error()
        for _ in range(2):
            got = torch.full_like(want, 0x66)
            torch.cuda.synchronize()  # the fill is done before the other stream writes
            tm.tiled_copy_noalloc(m, lst, got, stream=s)
            assert torch.equal(got, want)
