"""The one-GPU-only companion library (include/tmap_onegpu.h): the tensor-core GEMM whose B tile is
shared by the two CTAs of a cluster through TMA multicast ([H200-TMA] coolgpu "H200 · TMA" card,
§01 and §04 ③).  Opt-in: these tests build and load it themselves; nothing else does.

Every element of C within the fp32 summation bound K * 2^-23 * sum |a b| of the oracle's exact
dot product (as for stream_gemm); tensors that are not device memory of the current device are
refused with TM_EINVAL.
"""
import numpy as np
import pytest

import oracle
from gpu_util import guarded, to_host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def libs():
    import async_bulk_tensor_tmap_gb300 as tm  # raises if the CUDA library is missing
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from async_bulk_tensor_tmap_gb300 import onegpu  # builds the one-GPU library on first import
    return tm, onegpu


def bf16_normal(rows, cols, seed):
    v = np.random.default_rng(seed).standard_normal((rows, cols)).astype(np.float32)
    return ((v.view(np.uint32) + 0x7FFF + ((v.view(np.uint32) >> 16) & 1)) >> 16).astype(np.uint16)


def run(libs, a, b, stages=4, ldc=None):
    tm, onegpu = libs
    M, K = a.shape
    N = b.shape[0]
    ad = torch.from_numpy(a.reshape(-1).view(np.uint8).copy()).cuda()
    bd = torch.from_numpy(b.reshape(-1).view(np.uint8).copy()).cuda()
    ldc = N if ldc is None else ldc
    c = guarded(4 * M * ldc, 0xFF).view(torch.float32)  # all-ones bytes: a NaN in every float
    ma = tm.tmap_encode(tm.TM_BF16, ad, [K, M], [K * 2], [64, 128], swizzle=tm.TM_SWIZZLE_128B)
    mbh = tm.tmap_encode(tm.TM_BF16, bd, [K, N], [K * 2], [64, 128], swizzle=tm.TM_SWIZZLE_128B)
    onegpu.stream_gemm_multicast(ma, mbh, c, ldc=ldc, stages=stages)
    torch.cuda.synchronize()
    assert onegpu.tm_onegpu_check() == tm.TM_OK, onegpu.last_error()
    return to_host(c).reshape(M, ldc)


def within_bound(got, a, b):
    K = a.shape[1]
    exact = oracle.gemm(a, b)
    scale = oracle.gemm(a & 0x7FFF, b & 0x7FFF)  # sum of |products| (signs cleared)
    err = np.abs(got.astype(np.float64) - exact)
    return bool((err <= K * 2.0 ** -23 * scale).all())


@pytest.mark.parametrize("M,N,K", [(256, 512, 128), (128, 256, 64), (200, 300, 136),
                                   (384, 256, 320), (640, 768, 1024)])
def test_multicast_gemm_matches_oracle(libs, M, N, K):
    """Several clusters and tiles, ragged M / N / K, an odd number of 128-row tiles (the second CTA
    of the last cluster computes rows beyond M, which are not stored), K deep enough to wrap the
    ring."""
    a, b = bf16_normal(M, K, 21), bf16_normal(N, K, 22)
    got = run(libs, a, b)
    assert within_bound(got, a, b)
    assert np.isfinite(got).all()


@pytest.mark.parametrize("stages", [2, 3, 4])
def test_multicast_gemm_every_ring_depth(libs, stages):
    a, b = bf16_normal(256, 448, 23), bf16_normal(512, 448, 24)
    assert within_bound(run(libs, a, b, stages=stages), a, b)


def test_multicast_gemm_integer_inputs_are_exact_and_padding_kept(libs):
    """Small integers: every partial sum is an integer below 2^24, so the result is exact; a padded
    ldc leaves the padding columns untouched."""
    M, N, K = 384, 260, 192
    ai = (np.arange(M)[:, None] * 7 + np.arange(K)[None, :] * 3) % 9 - 4
    bi = (np.arange(N)[:, None] * 5 + np.arange(K)[None, :] * 11) % 7 - 3
    a = (ai.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    b = (bi.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    got = run(libs, a, b, ldc=264)
    np.testing.assert_array_equal(got[:, :N].astype(np.int64), ai @ bi.T)
    assert np.isnan(got[:, N:]).all()


def test_multicast_gemm_refuses_memory_of_no_device(libs):
    """Tensors in host memory (pinned or not) are not this GPU's memory: TM_EINVAL, nothing runs."""
    tm, onegpu = libs
    M = N = 256
    K = 64
    a = torch.zeros(M * K, dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(N * K, dtype=torch.bfloat16, device="cuda")
    ma = tm.tmap_encode(tm.TM_BF16, a, [K, M], [K * 2], [64, 128], swizzle=tm.TM_SWIZZLE_128B)
    mbh = tm.tmap_encode(tm.TM_BF16, b, [K, N], [K * 2], [64, 128], swizzle=tm.TM_SWIZZLE_128B)
    for c in (torch.zeros(M * N, dtype=torch.float32).pin_memory(),
              torch.zeros(M * N, dtype=torch.float32)):
        with pytest.raises(tm.TmapError) as e:
            onegpu.stream_gemm_multicast(ma, mbh, c)
        assert e.value.code == tm.TM_EINVAL
        assert "device memory of the current device" in str(e.value)
    host_b = torch.zeros(N * K, dtype=torch.bfloat16).pin_memory()
    mhost = tm.tmap_encode(tm.TM_BF16, host_b, [K, N], [K * 2], [64, 128], swizzle=tm.TM_SWIZZLE_128B)
    c = torch.zeros(M * N, dtype=torch.float32, device="cuda")
    with pytest.raises(tm.TmapError) as e:
        onegpu.stream_gemm_multicast(ma, mhost, c)
    assert e.value.code == tm.TM_EINVAL
    assert onegpu.tm_onegpu_check() == tm.TM_OK
