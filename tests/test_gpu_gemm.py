"""GPU parity of the ring in GEMM order with its tensor-core consumer, C = A * B^T (stream_gemm),
against the oracle (mlc.ai "Modern GPU Programming for MLSys", chapter "异步数据搬运：TMA", overview
and §"把 TMA 放进 pipeline").

Tolerance, from the arithmetic: the inputs are bf16, so every product is exact in fp32; whatever
order the tensor cores add the K products in, and whether they round to nearest or toward zero, a
sum of K terms in fp32 is within K * 2^-23 * sum |terms| of the exact sum.  Each element of C is
checked against that bound with the oracle's exact (double) sum and sum of |products|."""
import numpy as np
import pytest

import oracle
from gpu_util import guarded, to_host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def tm_lib():
    import async_bulk_tensor_tmap_gb300 as m  # raises if the CUDA library is missing
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return m


@pytest.fixture(params=["one_sm", "pair"])
def tm(request, tm_lib, monkeypatch):
    """The two forms of the consumer: one SM per 128-row tile; CTA pairs (tcgen05 cta_group::2,
    256-row tiles over two SMs)."""
    monkeypatch.setenv("TM_GEMM_PAIR", "1" if request.param == "pair" else "0")
    return tm_lib


def check(tm):
    torch.cuda.synchronize()
    rc = tm.tm_stream_check()
    assert rc == tm.TM_OK, tm.tm_last_error()


def bf16_normal(rows, cols, seed):
    v = np.random.default_rng(seed).standard_normal((rows, cols)).astype(np.float32)
    return ((v.view(np.uint32) + 0x7FFF + ((v.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)


def run(tm, a, b, stages=4, ldc=None):
    M, K = a.shape
    N = b.shape[0]
    ad = torch.from_numpy(a.reshape(-1).view(np.uint8).copy()).cuda()
    bd = torch.from_numpy(b.reshape(-1).view(np.uint8).copy()).cuda()
    ldc = N if ldc is None else ldc
    c = guarded(4 * M * ldc, 0xFF).view(torch.float32)  # all-ones bytes: a NaN in every float
    ma = tm.tmap_encode(tm.TM_BF16, ad, [K, M], [K * 2], [64, 128], swizzle=tm.TM_SWIZZLE_128B)
    mb = tm.tmap_encode(tm.TM_BF16, bd, [K, N], [K * 2], [64, 256], swizzle=tm.TM_SWIZZLE_128B)
    tm.stream_gemm(ma, mb, c, ldc=ldc, stages=stages)
    check(tm)
    return to_host(c).reshape(M, ldc)


def assert_within_bound(got, a, b, rows=None, cols=None):
    M, K = a.shape
    N = b.shape[0]
    rows = range(M) if rows is None else rows
    cols = range(N) if cols is None else cols
    worst = 0.0
    for m in rows:
        for n in cols:
            exact, scale = oracle.gemm_entry(a, b, m, n)
            bound = K * 2.0 ** -23 * scale
            err = abs(float(got[m, n]) - exact)
            assert err <= bound, (m, n, float(got[m, n]), exact, bound)
            worst = max(worst, err / bound if bound else 0.0)
    return worst


@pytest.mark.parametrize("M,N,K", [(256, 512, 128), (128, 256, 64), (200, 300, 136),
                                   (128, 256, 1024), (384, 256, 320)])
def test_gemm_matches_oracle(tm, M, N, K):
    a, b = bf16_normal(M, K, 1), bf16_normal(N, K, 2)
    got = run(tm, a, b)
    exact = oracle.gemm(a, b)
    scale = oracle.gemm(a & 0x7FFF, b & 0x7FFF)   # sum of |products| (signs cleared)
    bound = K * 2.0 ** -23 * scale
    err = np.abs(got.astype(np.float64) - exact)
    assert (err <= bound).all(), f"worst {float((err / bound).max()):.3g} of the bound"
    assert np.isfinite(got).all()


@pytest.mark.parametrize("stages", [2, 3, 4, 6, 7])
def test_gemm_every_ring_depth(tm, stages):
    a, b = bf16_normal(256, 448, 3), bf16_normal(512, 448, 4)
    got = run(tm, a, b, stages=stages)
    exact = oracle.gemm(a, b)
    scale = oracle.gemm(a & 0x7FFF, b & 0x7FFF)
    assert (np.abs(got - exact) <= 448 * 2.0 ** -23 * scale).all()


def test_gemm_integer_inputs_are_exact(tm):
    """Small integers: every partial sum is an integer below 2^24, so fp32 is exact in any order."""
    M, N, K = 128, 256, 192
    ai = (np.arange(M)[:, None] * 7 + np.arange(K)[None, :] * 3) % 9 - 4
    bi = (np.arange(N)[:, None] * 5 + np.arange(K)[None, :] * 11) % 7 - 3
    a = (ai.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    b = (bi.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    got = run(tm, a, b)
    np.testing.assert_array_equal(got.astype(np.int64), ai @ bi.T)


def test_gemm_padded_ldc_and_ragged_edges_leave_the_rest(tm):
    M, N, K = 130, 260, 72
    a, b = bf16_normal(M, K, 5), bf16_normal(N, K, 6)
    got = run(tm, a, b, ldc=264)
    assert np.isnan(got[:, N:]).all()          # padding columns untouched
    exact = oracle.gemm(a, b)
    scale = oracle.gemm(a & 0x7FFF, b & 0x7FFF)
    assert (np.abs(got[:, :N] - exact) <= K * 2.0 ** -23 * scale).all()


def test_gemm_last_wave_in_half_tiles(tm):
    """A C of 2 x 43 tiles of 256 x 256 (86 tiles over the 76 SM pairs of a 152-SM GB300): the pair
    form does the last 10 tiles as 256 x 128 halves; ragged M, N and K.  Every column of the split
    tiles (and their neighbours) for rows of both CTAs of both row tiles."""
    M, N, K = 500, 11000, 200
    a, b = bf16_normal(M, K, 11), bf16_normal(N, K, 12)
    got = run(tm, a, b, stages=7)
    rows = [0, 1, 127, 128, 255, 256, 300, 383, 384, 499]
    cols = list(range(9600, N))
    exact = oracle.gemm(a[rows], b[cols])
    scale = oracle.gemm(a[rows] & 0x7FFF, b[cols] & 0x7FFF)
    bound = K * 2.0 ** -23 * scale
    err = np.abs(got[rows][:, cols].astype(np.float64) - exact)
    assert (err <= bound).all(), float((err / np.maximum(bound, 1e-300)).max())
    assert np.isfinite(got).all()


def test_gemm_full_size_sampled(tm):
    """The benchmark's shape (M = N = 8192, K = 4096) in its launch configuration; sampled
    elements against the oracle, one by one (rows and columns of every tile position class)."""
    import workloads
    a, b = workloads.w7_operands()
    got = run(tm, a, b, stages=7)  # the bench's ring depth
    rng = np.random.default_rng(7)
    rows = sorted(set(rng.integers(0, 8192, 6).tolist()) | {0, 127, 128, 255, 256, 8191})
    cols = sorted(set(rng.integers(0, 8192, 6).tolist()) | {0, 255, 256, 8191})
    worst = assert_within_bound(got, a, b, rows, cols)
    print(f"worst error {worst:.3g} of the bound")
    assert np.isfinite(got).all()


def test_gemm_one_pair_tile(tm):
    """The smallest case of each form: one 256 x 256 tile, one k step."""
    a, b = bf16_normal(256, 64, 11), bf16_normal(256, 64, 12)
    got = run(tm, a, b)
    exact = oracle.gemm(a, b)
    scale = oracle.gemm(a & 0x7FFF, b & 0x7FFF)
    assert (np.abs(got - exact) <= 64 * 2.0 ** -23 * scale).all()
