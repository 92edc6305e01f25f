"""The quotient method of the NVFP4 quantiser, in exact rational arithmetic (no GPU).

The quantiser divides y = fl32(x S) by the E4M3 block scale sb without a division per value:
r = RN(1 / sb) once per block, then q0 = RN(y r), e = RN(y - sb q0) (an FMA) and
q = RN(q0 + e r) (another FMA), every step rounded to fp32 nearest-even.  Markstein's theorem
says that q is then RN(y / sb).  This file checks it where a wrong quotient would change an
E2M1 code: y within 12 fp32 steps of t sb for every E2M1 value and rounding midpoint t and
every finite positive E4M3 scale sb, both signs, each step computed exactly with Fractions
and rounded by a plain round-half-even to 24 significant bits."""
from fractions import Fraction

import numpy as np

E2M1_POINTS = [Fraction(t) for t in (0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0, 6.0)]


def rn32(x: Fraction) -> Fraction:
    """Round to the nearest fp32 value, ties to even (normal range)."""
    if x == 0:
        return Fraction(0)
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()   # floor(log2 a), within one
    if a < Fraction(2) ** e:
        e -= 1
    while a >= Fraction(2) ** (e + 1):
        e += 1
    m = a * Fraction(2) ** (23 - e)          # in [2^23, 2^24)
    n = m.numerator // m.denominator
    rest = m - n
    if rest > Fraction(1, 2) or (rest == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = Fraction(n) * Fraction(2) ** (e - 23)
    return r if x > 0 else -r


def e4m3_positive():
    vals = []
    for code in range(1, 0x7F):
        e, m = code >> 3, code & 7
        vals.append(Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7))
    return vals


def f32_neighbours(v: Fraction, k: int):
    """The fp32 values from k steps below RN(v) to k steps above it."""
    x = np.float32(float(rn32(v)))
    out = [x]
    lo = hi = x
    for _ in range(k):
        lo = np.nextafter(lo, np.float32(-np.inf))
        hi = np.nextafter(hi, np.float32(np.inf))
        out += [lo, hi]
    return [Fraction(float(t)) for t in out]


def test_rn32_matches_numpy_float32():
    rng = np.random.default_rng(7)
    for v in rng.standard_normal(200) * np.exp(rng.standard_normal(200) * 5):
        assert rn32(Fraction(float(v))) == Fraction(float(np.float32(v)))
    # ties go to the even significand: 1 + 2^-24 to 1, 1 + 3 * 2^-24 to 1 + 2^-22
    assert rn32(1 + Fraction(1, 2 ** 24)) == 1
    assert rn32(1 + Fraction(3, 2 ** 24)) == 1 + Fraction(2, 2 ** 23)


def test_fma_corrected_quotient_is_the_correctly_rounded_quotient():
    scales = e4m3_positive()
    assert len(scales) == 126 and max(scales) == 448
    checked = 0
    for sb in scales:
        r = rn32(1 / sb)
        for t in E2M1_POINTS:
            for y in f32_neighbours(t * sb, 12):
                for ys in (y, -y):
                    q0 = rn32(ys * r)
                    e = rn32(ys - sb * q0)
                    q = rn32(q0 + e * r)
                    assert q == rn32(ys / sb), (float(ys), float(sb))
                    checked += 1
    assert checked == 126 * len(E2M1_POINTS) * 25 * 2


def test_plain_reciprocal_product_is_not_enough():
    """The correction step matters: RN(y RN(1/sb)) misses the correctly rounded quotient for
    some of the same inputs (so the check above can fail)."""
    misses = 0
    for sb in e4m3_positive():
        r = rn32(1 / sb)
        for t in (Fraction(3, 4), Fraction(5, 4), Fraction(5, 2), Fraction(7, 2)):
            for y in f32_neighbours(t * sb, 2):
                misses += rn32(y * r) != rn32(y / sb)
    assert misses > 0
