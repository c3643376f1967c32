"""Pins for the oracle's scalar codecs (E4M3 block scales, E2M1 values).

Each check ties the oracle to something other than itself: torch's own
float8_e4m3fn conversion (a library routine), the bit-field definition of
E2M1, or an exhaustive comparison against exact rational rounding done by a
different method (threshold counting on exact float64 products).
"""

import numpy as np
import pytest
import torch

import oracle

# ----------------------------------------------------------------- helpers


def all_finite_bf16():
    """Every finite BF16 value as (uint16 bits, float64 value)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_to_f64(bits)
    keep = np.isfinite(vals)
    return bits[keep], vals[keep]


def e4m3_positive_finite():
    """The 126 positive finite E4M3 values (codes 0x01..0x7E) via torch."""
    codes = torch.arange(1, 0x7F, dtype=torch.uint8)
    return codes.numpy(), codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


# ----------------------------------------------------------------- E4M3


def test_e4m3_decode_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert (np.isnan(mine) == nan).all()
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.nanmax(mine) == 448.0 and oracle.e4m3_value(0x01) == 2.0**-9 and oracle.e4m3_value(0x08) == 2.0**-6


def test_e4m3_encode_matches_torch_on_every_bf16_below_464():
    bits, vals = all_finite_bf16()
    inrange = np.abs(vals) < 464.0
    x = vals[inrange].astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = oracle.e4m3_encode_many(x)
    assert np.array_equal(mine, ref)


def test_e4m3_encode_saturates_at_448():
    # torch's cast returns NaN from 464 up; the cache's codec saturates instead.
    for v in (464.0, 465.0, 1e4, 3.0e38):
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE
    assert oracle.e4m3_encode(448.0) == 0x7E and oracle.e4m3_encode(463.9) == 0x7E


def test_scale_rounding_equals_exact_rational_rounding_for_every_bf16_amax():
    """scale = E4M3(amax / 6), decided by the oracle on fl32(amax / 6), must equal
    the exact nearest-even E4M3 value of the rational amax / 6.  Exact method:
    amax / 6 >= midpoint  <=>  amax >= 6 * midpoint, and 6 * midpoint is exact
    in float64."""
    bits, vals = all_finite_bf16()
    amax = vals[(vals >= 0) & ~np.signbit(vals)]  # an amax is |x|: never -0
    codes, evals = e4m3_positive_finite()
    grid = np.concatenate([[0.0], evals])                  # code c <-> grid[c]
    mids = 0.5 * (grid[:-1] + grid[1:])                    # between code c and c+1
    above = amax[:, None] > 6.0 * mids[None, :]
    at = amax[:, None] == 6.0 * mids[None, :]
    exact = above.sum(axis=1)
    # a tie goes to the even code of its pair
    tie_idx = np.nonzero(at.any(axis=1))[0]
    for i in tie_idx:
        c = int(np.nonzero(at[i])[0][0])
        exact[i] = c if c % 2 == 0 else c + 1
    exact = np.minimum(exact, 0x7E)
    mine = oracle.e4m3_encode_many((amax.astype(np.float32) / np.float32(6.0)).astype(np.float32))
    assert len(tie_idx) > 0  # there are exact ties among BF16 amax values
    assert np.array_equal(mine, exact.astype(np.uint8))


# ----------------------------------------------------------------- E2M1


def test_e2m1_decode_from_bit_fields():
    """E2M1: bit 3 sign, bits 2..1 exponent with bias 1, bit 0 mantissa;
    exponent 0 is subnormal (0.m x 2^0)."""
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = (m * 0.5) if e == 0 else (2.0 ** (e - 1)) * (1.0 + 0.5 * m)
        expect = -mag if s else mag
        got = oracle.e2m1_value(code)
        assert got == expect and np.signbit(got) == bool(s)
    assert sorted({abs(oracle.e2m1_value(c)) for c in range(16)}) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


@pytest.mark.parametrize("x,code", [
    (0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),   # ties -> even code
    (0.2499, 0), (0.2501, 1), (5.0001, 7), (6.0, 7), (6.5, 7), (1e30, 7),       # nearest, saturate
    (-0.1, 8), (-0.0, 8), (0.0, 0), (-5.0, 14),                                  # sign kept
])
def test_e2m1_rounding_special_cases(x, code):
    assert oracle.e2m1_encode(x) == code


def test_e2m1_decision_equals_exact_rational_rounding_over_all_bf16_and_scales():
    """For every finite BF16 x and every positive finite E4M3 scale d, the
    oracle's code E2M1(fl32(x / d)) must equal exact nearest-even rounding of
    the rational x / d.  Exact method: count the midpoints m with |x| > m*d
    (m*d has at most 3 + 4 significant bits, exact in float64), resolving
    |x| == m*d to the even code."""
    bits, vals = all_finite_bf16()
    _, scales = e4m3_positive_finite()
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    # Ties go to the even code: at midpoint k (between codes k and k+1) pick even.
    tie_code = np.array([0, 2, 2, 4, 4, 6, 6], dtype=np.uint8)
    ax = np.abs(vals)
    neg = np.signbit(vals)
    n_ties = 0
    for d in scales:
        thr = mids * d
        mag = (ax[:, None] > thr[None, :]).sum(axis=1).astype(np.uint8)
        at = ax[:, None] == thr[None, :]
        hit = at.any(axis=1)
        n_ties += int(hit.sum())
        mag[hit] = tie_code[np.argmax(at[hit], axis=1)]
        exact = np.where(neg, mag | 8, mag).astype(np.uint8)
        mine = oracle.e2m1_encode_quotients(vals.astype(np.float32), np.float32(d))
        assert np.array_equal(mine, exact), "scale %r" % d
    assert n_ties > 1000
