"""The FP8 dispatch kernel forms fl(v / s) with one multiply and one
Markstein correction (P. Markstein, IBM J. Res. Dev. 34(1), 1990) instead of
an IEEE division.  That is only exact because the operands are narrow: v is a
bf16 value (significand V of at most 8 bits) and the block scale is
s = fl(amax / 448) = fl(M / 7) * 2^j for the 8-bit significand M of a bf16
amax ("FP8 e4m3 with 1x128 block scales", scale = amax / 448).  Every step
scales exactly with powers of two, so the (V, M) pairs are all the cases.

These tests redo the kernel's arithmetic on every pair in exact rational
arithmetic, rounding each step to fp32 by hand, and compare with the
correctly rounded quotient.  No GPU, no oracle: this checks the method the
kernel relies on, not an implementation of it."""
from fractions import Fraction as F

import pytest


def rn32(x: F) -> F:
    """x rounded to the nearest fp32 value, ties to even (normal range)."""
    if x == 0:
        return F(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if F(2) ** e > a:
        e -= 1
    scaled = a / F(2) ** (e - 23)  # in [2^23, 2^24)
    n, rem = divmod(scaled.numerator, scaled.denominator)
    rem = F(rem, scaled.denominator)
    if rem > F(1, 2) or (rem == F(1, 2) and n % 2 == 1):
        n += 1
    return sign * F(n) * F(2) ** (e - 23)


def kernel_quotients(V: int, M: int):
    """q0 = RN(v y) and q1 = RN(q0 - RN(s q0 - v) y) with s = fl(M/7),
    y = RN(1/s), exactly as the kernel sequences them (fma = one rounding)."""
    s = rn32(F(M, 7))
    y = rn32(1 / s)
    q0 = rn32(V * y)
    r = rn32(s * q0 - V)
    q1 = rn32(q0 - r * y)
    return s, q0, q1


def test_rn32_matches_numpy_float32():
    """rn32 against numpy's float64 -> float32 conversion (one correct
    rounding) on values exactly representable in float64: random 53-bit
    integers times powers of two, and exact ties between fp32 neighbours."""
    np = pytest.importorskip("numpy")
    rng = np.random.default_rng(0)
    cases = [int(n) for n in rng.integers(1, 1 << 53, size=400, dtype=np.int64)]
    cases += [((1 << 24) + 2 * i + 1) << 5 for i in range(50)]  # ties, both parities
    cases += [(1 << 24) - 1, 1 << 24, (1 << 24) + 1, (1 << 25) + 3]
    for n in cases:
        for e in (-140, -60, -20, 0, 30):
            x = F(n) * F(2) ** e
            want = F(float(np.float32(np.float64(n) * np.float64(2.0) ** e)))
            assert rn32(x) == want, (n, e)
            assert rn32(-x) == -want


def test_one_correction_is_exact_for_every_significand_pair():
    wrong_q0 = 0
    for M in range(128, 256):
        for V in range(1, 256):
            s, q0, q1 = kernel_quotients(V, M)
            exact = rn32(F(V) / s)
            assert q1 == exact, (V, M)
            wrong_q0 += q0 != exact
    # the correction is needed: RN(v y) alone misses for a quarter of the pairs
    assert wrong_q0 > 0.2 * 128 * 255


def test_scale_table_identity():
    """fl(m / 448) = fl(M / 7) * 2^(k - 6) and RN(1/s) = RN(1/fl(M/7)) * 2^(6 - k)
    for m = M * 2^k: the kernel's 128-entry tables."""
    for M in range(128, 256):
        for k in (-60, -7, 0, 5, 40):
            m = F(M) * F(2) ** k
            s = rn32(m / 448)
            assert s == rn32(F(M, 7)) * F(2) ** (k - 6)
            assert rn32(1 / s) == rn32(1 / rn32(F(M, 7))) * F(2) ** (6 - k)
