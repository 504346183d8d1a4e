"""Pins of the oracle's GEMM consumer of the k-ordered ring, C = A * B^T for bf16 A (M x K) and
B (N x K) -- mlc.ai "Modern GPU Programming for MLSys", chapter "异步数据搬运：TMA", overview and
§"把 TMA 放进 pipeline": the tensor cores consume the A and B tiles of step k while TMA loads those
of step k + 1.  The oracle returns each C element as a double; these pins check it against exact
integer and rational arithmetic written here, not against itself."""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Values exactly representable in bf16 -> their bit patterns."""
    f = np.asarray(x, np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert ((bits.astype(np.uint32) << 16).view(np.float32) == f).all(), "not a bf16 value"
    return bits


def bf16_value(h: int) -> Fraction:
    return Fraction(float(np.array([h << 16], np.uint32).view(np.float32)[0]))


@pytest.mark.parametrize("m,n,k", [(7, 9, 1), (13, 11, 37), (20, 17, 300)])
def test_small_integers_are_exact(m, n, k):
    ai = [[(r * 7 + c * 3) % 9 - 4 for c in range(k)] for r in range(m)]
    bi = [[(r * 5 + c * 11) % 7 - 3 for c in range(k)] for r in range(n)]
    a, b = bf16_bits(np.array(ai, np.float32)), bf16_bits(np.array(bi, np.float32))
    got = oracle.gemm(a, b)
    for r in range(m):
        for c in range(n):
            assert got[r, c] == sum(ai[r][i] * bi[c][i] for i in range(k)), (r, c)


def test_one_hot_rows_pick_entries_of_b():
    k = 64
    a = bf16_bits(np.eye(16, k, dtype=np.float32))           # A[m][k] = 1 iff k == m
    rng = np.random.default_rng(1)
    bv = rng.standard_normal((24, k)).astype(np.float32)
    b = bf16_bits((bv.view(np.uint32) & 0xFFFF0000).view(np.float32))
    got = oracle.gemm(a, b)
    want = (b.astype(np.uint32) << 16).view(np.float32)[:, :16].T   # C[m][n] = B[n][m]
    np.testing.assert_array_equal(got, want.astype(np.float64))


def test_random_bf16_against_exact_rationals():
    rng = np.random.default_rng(2)
    m, n, k = 5, 6, 257
    # wide exponent range: a float32 accumulator would lose these low-order terms
    a = bf16_bits(((rng.standard_normal((m, k)) * np.exp2(rng.integers(-20, 20, (m, k))))
                   .astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32))
    b = bf16_bits(((rng.standard_normal((n, k)) * np.exp2(rng.integers(-20, 20, (n, k))))
                   .astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32))
    got = oracle.gemm(a, b)
    for r in range(m):
        for c in range(n):
            terms = [bf16_value(int(a[r, i])) * bf16_value(int(b[c, i])) for i in range(k)]
            exact = sum(terms)
            scale = sum(abs(t) for t in terms)
            assert abs(Fraction(got[r, c]) - exact) <= scale * Fraction(k, 2 ** 52), (r, c)
            v, s = oracle.gemm_entry(a, b, r, c)
            assert v == got[r, c] and abs(Fraction(s) - scale) <= scale * Fraction(k, 2 ** 52)


def test_swapping_operands_transposes():
    rng = np.random.default_rng(3)
    a = bf16_bits(((rng.standard_normal((9, 40)).astype(np.float32).view(np.uint32)
                    & 0xFFFF0000).view(np.float32)))
    b = bf16_bits(((rng.standard_normal((12, 40)).astype(np.float32).view(np.uint32)
                    & 0xFFFF0000).view(np.float32)))
    np.testing.assert_array_equal(oracle.gemm(a, b), oracle.gemm(b, a).T)


def test_blocks_and_leading_k():
    rng = np.random.default_rng(4)
    a = rng.integers(0, 1 << 16, (30, 50), dtype=np.uint64).astype(np.uint16) & 0x3F7F
    b = rng.integers(0, 1 << 16, (20, 50), dtype=np.uint64).astype(np.uint16) & 0x3F7F
    full = oracle.gemm(a, b)
    np.testing.assert_array_equal(oracle.gemm(a, b, 4, 17, 3, 11), full[4:17, 3:11])
    # the first 31 columns of K only: same as slicing the operands
    np.testing.assert_array_equal(oracle.gemm(a, b, k=31),
                                  oracle.gemm(np.ascontiguousarray(a[:, :31]),
                                              np.ascontiguousarray(b[:, :31])))
