"""Pins of the oracle's general reduce (add / min / max over f32, f16, bf16, u32, s32) against
library routines and exact rational arithmetic -- fangpin "gpu-hpc-book" ch. 08 "Cuda TMA",
§"TMA reduce，把“搬运”和“归约”合并" (the write-back combines each element with global memory by add,
min and the like).  The pages fix no rounding for 16-bit float adds; this library reads it as the
exact sum rounded to nearest, ties to even, which these pins check independently."""
from fractions import Fraction

import numpy as np
import pytest

import oracle

F32, F16, BF16, U32, S32 = oracle.F32, oracle.F16, oracle.BF16, oracle.U32, oracle.S32
ADD, MIN, MAX = oracle.ADD, oracle.MIN, oracle.MAX


def bf16_value(h: int) -> Fraction:
    return Fraction(float(np.array([h << 16], np.uint32).view(np.float32)[0]))


def bf16_round_exact(x: Fraction) -> int:
    """x rounded to bfloat16 (8 significand bits, exponents -126..127, subnormals, overflow to
    infinity), ties to even, with exact rational arithmetic."""
    sign = 0x8000 if x < 0 else 0
    x = abs(x)
    if x == 0:
        return sign
    e = x.numerator.bit_length() - x.denominator.bit_length()
    if Fraction(2) ** e > x:
        e -= 1                      # now 2^e <= x < 2^(e+1)
    e = max(e, -126)
    q = Fraction(2) ** (e - 7)
    n = round(x / q)                # Fraction rounding: half to even
    if n >= 256:
        n //= 2
        e += 1
    if e > 127:
        return sign | 0x7F80
    if n < 128:
        return sign | n             # subnormal
    return sign | ((e + 127) << 7) | (n - 128)


def random_bf16(rng, n):
    """Finite bf16 patterns with exponents spread over a wide range."""
    mant = rng.integers(0, 128, n)
    exp = rng.integers(1, 255, n)
    sign = rng.integers(0, 2, n)
    return (sign << 15) | (exp << 7) | mant


def test_bf16_add_is_correctly_rounded():
    rng = np.random.default_rng(1)
    a = random_bf16(rng, 3000)
    # partners near a (small exponent differences: most rounding happens here) and far from it
    b_near = (a & 0x8000) ^ (rng.integers(0, 2, 3000) << 15) | \
        (np.clip(((a >> 7) & 0xFF) + rng.integers(-9, 10, 3000), 1, 254) << 7) | rng.integers(0, 128, 3000)
    b_far = random_bf16(rng, 3000)
    for x, y in list(zip(a, b_near)) + list(zip(a, b_far)):
        x, y = int(x), int(y)
        want = bf16_round_exact(bf16_value(x) + bf16_value(y))
        assert oracle.combine(x, y, BF16, ADD) == want, (hex(x), hex(y))


def test_bf16_add_ties_go_to_even():
    one = 0x3F80                      # 1.0
    half_ulp = bf16_round_exact(Fraction(1, 256))   # 2^-8: exactly half an ulp of 1.0
    assert oracle.combine(one, half_ulp, BF16, ADD) == one           # 1 + 2^-8 -> 1 (even)
    three_halves_ulp = bf16_round_exact(Fraction(3, 256))
    assert oracle.combine(one, three_halves_ulp, BF16, ADD) == one + 2  # 1 + 3*2^-8 -> 1 + 2^-6


def test_f16_add_matches_numpy_half():
    rng = np.random.default_rng(2)
    bits = rng.integers(0, 1 << 16, 20000).astype(np.uint16)
    bits = bits[(bits & 0x7C00) != 0x7C00]
    a, b = bits[0::2][:8000], bits[1::2][:8000]
    fa = a.view(np.float16).astype(np.float64)
    fb = b.view(np.float16).astype(np.float64)
    with np.errstate(over="ignore"):
        want = (fa + fb).astype(np.float16).view(np.uint16)   # the f16 double sum is exact
    for x, y, w in zip(a, b, want):
        assert oracle.combine(int(x), int(y), F16, ADD) == int(w), (hex(x), hex(y))


def test_f16_special_cases():
    h = lambda v: int(np.float16(v).view(np.uint16))
    assert oracle.combine(h(65504.0), h(16.0), F16, ADD) == 0x7C00          # ties to even -> inf
    assert oracle.combine(h(65504.0), h(8.0), F16, ADD) == h(65504.0)
    sub = 0x0001                                                            # 2^-24
    assert oracle.combine(sub, sub, F16, ADD) == 0x0002                     # subnormals kept
    assert oracle.combine(h(1.0), h(-1.0), F16, ADD) == 0x0000


def test_f32_ops_match_numpy():
    rng = np.random.default_rng(3)
    a = rng.standard_normal(5000).astype(np.float32)
    b = (rng.standard_normal(5000) * 3).astype(np.float32)
    ua, ub = a.view(np.uint32), b.view(np.uint32)
    for op, ref in ((ADD, a + b), (MIN, np.minimum(a, b)), (MAX, np.maximum(a, b))):
        ref = ref.astype(np.float32).view(np.uint32)
        got = np.array([oracle.combine(int(x), int(y), F32, op) for x, y in zip(ua, ub)], np.uint32)
        np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("t", [F16, BF16])
def test_half_min_max_match_numpy(t):
    rng = np.random.default_rng(4 + t)
    v = rng.standard_normal(4000).astype(np.float32)
    if t == F16:
        bits = v.astype(np.float16).view(np.uint16)
        vals = bits.view(np.float16).astype(np.float64)
    else:
        bits = (v.view(np.uint32) >> 16).astype(np.uint16)
        vals = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    a, b, fa, fb = bits[0::2], bits[1::2], vals[0::2], vals[1::2]
    for op, pick in ((MIN, np.where(fb < fa, b, a)), (MAX, np.where(fb > fa, b, a))):
        got = np.array([oracle.combine(int(x), int(y), t, op) for x, y in zip(a, b)], np.uint16)
        np.testing.assert_array_equal(got, pick)


def test_integer_ops_match_numpy():
    rng = np.random.default_rng(5)
    a = rng.integers(0, 1 << 32, 5000, dtype=np.uint64).astype(np.uint32)
    b = rng.integers(0, 1 << 32, 5000, dtype=np.uint64).astype(np.uint32)
    sa, sb = a.view(np.int32), b.view(np.int32)
    cases = [(U32, ADD, a + b), (U32, MIN, np.minimum(a, b)), (U32, MAX, np.maximum(a, b)),
             (S32, ADD, (sa + sb).view(np.uint32)), (S32, MIN, np.minimum(sa, sb).view(np.uint32)),
             (S32, MAX, np.maximum(sa, sb).view(np.uint32))]
    for t, op, ref in cases:
        got = np.array([oracle.combine(int(x), int(y), t, op) for x, y in zip(a, b)], np.uint32)
        np.testing.assert_array_equal(got, ref, err_msg=f"type {t} op {op}")


@pytest.mark.parametrize("t,op", [(BF16, ADD), (F16, MAX), (S32, MIN), (U32, ADD)])
def test_tile_reduce_equals_elementwise(t, op):
    """Over a ragged box grid with a swizzled image in between, every in-bounds element gets
    exactly one combine and nothing else changes."""
    rng = np.random.default_rng(6 + op)
    es = oracle.TYPE_ESIZE[t]
    rows, cols, pitch = 70, 40 if es == 4 else 72, 48 if es == 4 else 80
    span, box0 = (128, 32) if es == 4 else (128, 64)
    dst = rng.integers(0, 1 << 16, (rows, pitch)).astype(np.uint16 if es == 2 else np.uint32)
    src = rng.integers(0, 1 << 16, (rows, pitch)).astype(dst.dtype)
    if t in (F16, BF16):  # keep floats finite
        dst &= 0xBBFF
        src &= 0xBBFF
    r = dict(dims=[cols, rows], strides=[pitch * es], box=[box0, 16])
    want = dst.copy()
    for i in range(rows):
        for j in range(cols):
            want[i, j] = oracle.combine(int(dst[i, j]), int(src[i, j]), t, op)
    md = oracle.Map(dst, es, r["dims"], r["strides"], r["box"], span)
    ms = oracle.Map(src, es, r["dims"], r["strides"], r["box"], span)
    oracle.tile_reduce(md, ms, t, op)
    np.testing.assert_array_equal(dst, want)


def _is_nan(bits: int, t: int) -> bool:
    if t == F32:
        return (bits & 0x7F800000) == 0x7F800000 and (bits & 0x007FFFFF) != 0
    if t == F16:
        return (bits & 0x7C00) == 0x7C00 and (bits & 0x03FF) != 0
    return (bits & 0x7F80) == 0x7F80 and (bits & 0x007F) != 0


# IEEE 754 facts of one correctly rounded add (round to nearest): infinities absorb finite values,
# opposite infinities and NaN operands give a NaN, overflow rounds to infinity, x + (-x) is +0,
# (-0) + (-0) is -0, and subnormal sums are exact.  NaN stands for any NaN pattern.
NAN = None
SPECIAL_ADDS = {
    F32: [(0x7F800000, 0x3F800000, 0x7F800000), (0xFF800000, 0x3F800000, 0xFF800000),
          (0x7F800000, 0xFF800000, NAN), (0x7FC00000, 0x3F800000, NAN), (0x3F800000, 0x7FC00000, NAN),
          (0x7F7FFFFF, 0x7F7FFFFF, 0x7F800000), (0xFF7FFFFF, 0xFF7FFFFF, 0xFF800000),
          (0x00000001, 0x00000001, 0x00000002), (0x00800000, 0x80000001, 0x007FFFFF),
          (0x3F800000, 0xBF800000, 0x00000000), (0x80000000, 0x80000000, 0x80000000),
          (0x00000000, 0x80000000, 0x00000000), (0x807FFFFF, 0x00000001, 0x807FFFFE)],
    F16: [(0x7C00, 0x3C00, 0x7C00), (0xFC00, 0x3C00, 0xFC00), (0x7C00, 0xFC00, NAN),
          (0x7E00, 0x3C00, NAN), (0x3C00, 0x7E00, NAN), (0x7BFF, 0x7BFF, 0x7C00),
          (0xFBFF, 0xFBFF, 0xFC00), (0x0001, 0x0001, 0x0002), (0x0400, 0x8001, 0x03FF),
          (0x3C00, 0xBC00, 0x0000), (0x8000, 0x8000, 0x8000), (0x0000, 0x8000, 0x0000),
          (0x03FF, 0x0001, 0x0400)],
    BF16: [(0x7F80, 0x3F80, 0x7F80), (0xFF80, 0x3F80, 0xFF80), (0x7F80, 0xFF80, NAN),
           (0x7FC0, 0x3F80, NAN), (0x3F80, 0x7FC0, NAN), (0x7F7F, 0x7F7F, 0x7F80),
           (0xFF7F, 0xFF7F, 0xFF80), (0x0001, 0x0001, 0x0002), (0x0080, 0x8001, 0x007F),
           (0x3F80, 0xBF80, 0x0000), (0x8000, 0x8000, 0x8000), (0x0000, 0x8000, 0x0000),
           (0x007F, 0x0001, 0x0080)],
}


@pytest.mark.parametrize("t", [F32, F16, BF16])
def test_special_value_adds_follow_ieee(t):
    for a, b, want in SPECIAL_ADDS[t]:
        got = oracle.combine(a, b, t, ADD)
        if want is NAN:
            assert _is_nan(got, t), (hex(a), hex(b), hex(got))
        else:
            assert got == want, (hex(a), hex(b), hex(got), hex(want))


@pytest.mark.parametrize("t, one, nan, pz, nz", [(F32, 0x3F800000, 0x7FC00000, 0, 0x80000000),
                                                (F16, 0x3C00, 0x7E00, 0, 0x8000),
                                                (BF16, 0x3F80, 0x7FC0, 0, 0x8000)])
def test_special_value_min_max_keep_dst_unless_src_is_strictly_beyond(t, one, nan, pz, nz):
    # src replaces dst only when it compares strictly below (min) / above (max): a NaN on either
    # side and a tie of +0 with -0 keep dst
    for op in (MIN, MAX):
        assert oracle.combine(nan, one, t, op) == nan
        assert oracle.combine(one, nan, t, op) == one
        assert oracle.combine(pz, nz, t, op) == pz
        assert oracle.combine(nz, pz, t, op) == nz
    assert oracle.combine(one, nz, t, MIN) == nz
    assert oracle.combine(nz, one, t, MAX) == one


def test_f16_adds_with_every_special_exponent_match_numpy():
    """All f16 patterns, infinities and NaNs included, against numpy's half add (the double sum
    of two halves is exact, so numpy's rounding of it is the reference); NaN results as NaN."""
    rng = np.random.default_rng(9)
    specials = np.array([0x7C00, 0xFC00, 0x7E00, 0xFE01, 0x0000, 0x8000, 0x0001, 0x83FF, 0x7BFF,
                         0xFBFF, 0x0400], np.uint16)
    a = np.concatenate([np.repeat(specials, len(specials)), rng.integers(0, 1 << 16, 4000).astype(np.uint16)])
    b = np.concatenate([np.tile(specials, len(specials)), rng.integers(0, 1 << 16, 4000).astype(np.uint16)])
    with np.errstate(over="ignore", invalid="ignore"):
        ref = (a.view(np.float16).astype(np.float64) + b.view(np.float16).astype(np.float64)).astype(np.float16)
    for x, y, r in zip(a, b, ref):
        got = oracle.combine(int(x), int(y), F16, ADD)
        if np.isnan(r):
            assert _is_nan(got, F16), (hex(x), hex(y), hex(got))
        else:
            assert got == int(r.view(np.uint16)), (hex(x), hex(y), hex(got))
