"""The quantisers' quotient without a GPU: the fp32 steps the kernels take for
x / den (den >= 2^-92) -- y = RN(1/den), q = RN(x y), then twice q <- RN(q + RN(x - q den) y)
with each inner product-and-subtract one FMA, the sign of x kept -- emulated here in exact
rational arithmetic with one rounding per operation, give the correctly rounded quotient:
the same fp32 value as IEEE division.  Cases sit on and one ulp around e2m1 and e4m3
rounding midpoints (where a quotient one ulp off would change a code), plus random pairs
and zeros of both signs.  The GPU tests compare the kernels' codes with the oracle's; this
pins the arithmetic those kernels rely on."""
import math
import random
from fractions import Fraction

import numpy as np


def rn32(v: Fraction) -> float:
    """v rounded to the nearest fp32 value, ties to even (normal and subnormal range)."""
    if v == 0:
        return 0.0
    sign = -1.0 if v < 0 else 1.0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 23)
    m = a / ulp
    f = m.numerator // m.denominator
    r = m - f
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return sign * float(f * ulp)


def fma_quotient(x: float, den: float) -> float:
    y = rn32(Fraction(1) / Fraction(den))
    q = rn32(Fraction(x) * Fraction(y))
    for _ in range(2):
        r = rn32(Fraction(x) - Fraction(q) * Fraction(den))
        q = rn32(Fraction(q) + Fraction(r) * Fraction(y))
    return math.copysign(abs(q), x)


def ieee(x: float, den: float) -> float:
    return float(np.float32(x) / np.float32(den))


def same(a: float, b: float) -> bool:
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


def midpoints():
    e2m1 = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    e4m3 = [(1 + (m + 0.5) / 8) * 2.0 ** e for e in range(-6, 9) for m in range(8)]
    e4m3 += [(m + 0.5) * 2.0 ** -9 for m in range(8)]
    return e2m1 + e4m3


def test_quotient_near_rounding_midpoints():
    rng = random.Random(3)
    mids = midpoints()
    n = 0
    for _ in range(600):
        den = float(np.float32(2.0 ** rng.uniform(-92, 40) * rng.uniform(1, 2)))
        if den < 2.0 ** -92:
            continue
        x0 = rn32(Fraction(rng.choice(mids) * rng.choice([-1, 1])) * Fraction(den))
        for x in (x0, float(np.nextafter(np.float32(x0), np.float32(np.inf))),
                  float(np.nextafter(np.float32(x0), np.float32(-np.inf)))):
            assert same(fma_quotient(x, den), ieee(x, den)), (x, den)
            n += 1
    assert n > 1500


def test_quotient_random_and_signed_zeros():
    rng = random.Random(4)
    for _ in range(600):
        den = float(np.float32(2.0 ** rng.uniform(-92, 60) * rng.uniform(1, 2)))
        if den < 2.0 ** -92:
            continue
        x = float(np.float32(den * rng.uniform(-8, 8) * 2.0 ** rng.choice([0, 0, -3, -12])))
        assert same(fma_quotient(x, den), ieee(x, den)), (x, den)
    for den in (1.0, 3.0, 0.1, 2.0 ** -92):
        den = float(np.float32(den))
        assert same(fma_quotient(0.0, den), 0.0)
        assert same(fma_quotient(-0.0, den), -0.0)


def test_uncorrected_product_is_not_enough():
    """Without the correction steps, RN(x RN(1/den)) is one ulp off for many quotients near
    midpoints (about a quarter of such cases here): the pins above depend on the steps.  (One
    step already matched every case tried; the kernels take a second as a margin.)"""
    rng = random.Random(5)
    mids = midpoints()
    off = 0
    for _ in range(3000):
        den = float(np.float32(2.0 ** rng.uniform(-60, 40) * rng.uniform(1, 2)))
        x = rn32(Fraction(rng.choice(mids)) * Fraction(den))
        y = rn32(Fraction(1) / Fraction(den))
        q = rn32(Fraction(x) * Fraction(y))
        if q != ieee(x, den):
            off += 1
    assert off > 0
