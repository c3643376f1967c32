"""Exact rational rounding for the oracle's tensor-scale pins (fractions.Fraction).

Written from the format definitions alone, independently of the oracle's C:
  * E2M1 magnitudes {0, 1/2, 1, 3/2, 2, 3, 4, 6}; E4M3 (OCP "fn") magnitudes of
    codes 0..126 from their bit fields (subnormals m 2^-9, normals
    (8 + m) 2^(e - 10)); rounding to nearest, ties to the even code,
    saturating at the largest value;
  * BF16: 8 significant bits from 2^-126 up, steps of 2^-133 below, infinity
    once the rounded magnitude reaches 2^128; nearest, ties to even.
"""

from fractions import Fraction as Fr

import numpy as np

E2M1 = [Fr(0), Fr(1, 2), Fr(1), Fr(3, 2), Fr(2), Fr(3), Fr(4), Fr(6)]


def _e4m3(c):
    e, m = (c >> 3) & 15, c & 7
    return Fr(m, 512) if e == 0 else Fr(8 + m) * Fr(2) ** (e - 10)


E4M3 = [_e4m3(c) for c in range(127)]


def rne_code(q: Fr, vals) -> int:
    """Index of the nearest of the ascending magnitudes vals to q >= 0, ties
    to the even index, saturating at the last."""
    if q >= vals[-1]:
        return len(vals) - 1
    hi = next(i for i, v in enumerate(vals) if v >= q)
    if vals[hi] == q:
        return hi
    lo = hi - 1
    mid = (vals[lo] + vals[hi]) / 2
    if q != mid:
        return lo if q < mid else hi
    return lo if lo % 2 == 0 else hi


def frac_of_f32(x) -> Fr:
    return Fr(float(np.float32(x)))


def floor_log2(a: Fr) -> int:
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fr(2) ** e > a:
        e -= 1
    while Fr(2) ** (e + 1) <= a:
        e += 1
    return e


def bf16_rne_bits(x: Fr) -> int:
    """BF16 bit pattern of the real x rounded once to nearest-even."""
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    if a == 0:
        return sign
    e = floor_log2(a)
    step = Fr(2) ** (e - 7) if e >= -126 else Fr(2) ** -133
    k = a / step
    f = k.numerator // k.denominator
    r = k - f
    if r > Fr(1, 2) or (r == Fr(1, 2) and f % 2 == 1):
        f += 1
    v = f * step
    if v >= Fr(2) ** 128:
        return sign | 0x7F80
    if v < Fr(2) ** -126:
        return sign | f
    ve = floor_log2(v)
    mant = v / Fr(2) ** ve * 128 - 128
    assert mant.denominator == 1
    return sign | ((ve + 127) << 7) | int(mant)


def bf16_value(bits: int) -> Fr:
    return Fr(float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0]))


def bf16_neighbours(t: Fr, k: int = 1):
    """Finite positive BF16 values around the positive real t: the nearest ones
    below and above it and k more on each side (as bit patterns)."""
    b = bf16_rne_bits(t) & 0x7FFF
    out = set()
    for d in range(-k - 1, k + 2):
        c = b + d
        if 0 < c < 0x7F80:
            out.add(c)
    return sorted(out)
