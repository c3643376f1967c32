"""Pins of the oracle's tensor-scale calibration (g = amax / (6 * 448), the
two-level NVFP4 rule for the FP32 tensor scale that the page fixes at 1.0 and
names as the thing to calibrate): closed forms, exact rational rounding, the
link to the block quantiser (the block holding amax gets E4M3's largest scale
and no scale saturates), and the error bound it buys on large activations."""

from fractions import Fraction

import numpy as np

import oracle
from oracle_helpers import bf16_bits_to_f64, to_bf16_bits


def _with_planted(rng, value, n=4096):
    x = rng.uniform(-1.0, 1.0, size=n).astype(np.float32)
    x[int(rng.integers(n))] = value
    return to_bf16_bits(x)


def test_closed_forms():
    rng = np.random.default_rng(5)
    assert oracle.calibrate_global_scale(_with_planted(rng, 5376.0)) == np.float32(2.0)
    assert oracle.calibrate_global_scale(_with_planted(rng, -5376.0)) == np.float32(2.0)
    assert oracle.calibrate_global_scale(_with_planted(rng, 2688.0)) == np.float32(1.0)
    assert oracle.calibrate_global_scale(_with_planted(rng, 2688.0 / 1024)) == np.float32(2.0**-10)
    assert oracle.calibrate_global_scale(np.zeros(64, dtype=np.uint16)) == np.float32(1.0)
    assert oracle.calibrate_global_scale(np.array([0x8000] * 8, dtype=np.uint16)) == np.float32(1.0)  # -0
    assert oracle.calibrate_global_scale(np.zeros(0, dtype=np.uint16)) == np.float32(1.0)


def test_infinities_and_nans_are_ignored():
    x = np.array([0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x4528], dtype=np.uint16)  # +inf, -inf, nan, nan, 2688
    assert oracle.calibrate_global_scale(x) == np.float32(1.0)


def test_result_is_the_correctly_rounded_fp32_quotient():
    rng = np.random.default_rng(6)
    for _ in range(200):
        x = to_bf16_bits(rng.standard_normal(256) * np.exp(rng.uniform(-20, 20)))
        amax = Fraction(float(np.abs(bf16_bits_to_f64(x)).max()))
        g = oracle.calibrate_global_scale(x)
        exact = amax / 2688
        # g is the FP32 value nearest to amax / 2688: within half an FP32 ulp of it
        gf = Fraction(float(g))
        ulp = Fraction(2.0 ** (np.floor(np.log2(float(g))) - 23))
        assert abs(gf - exact) <= ulp / 2


def _quantise_tensor(x_bits, g):
    """(scale values, dequantised values) of every 16-block, via the oracle's quantiser."""
    blocks = x_bits.reshape(-1, 16)
    scales, deq = [], []
    for blk in blocks:
        codes, sc = oracle.quantize_block16(blk, g)
        s = oracle.e4m3_value(sc)
        scales.append(s)
        deq.append([oracle.e2m1_value(c) * s * float(np.float32(g)) for c in codes])
    return np.array(scales), np.array(deq)


def test_calibrated_scale_fills_e4m3_range_without_saturating():
    rng = np.random.default_rng(7)
    for mag in (1e-6, 1.0, 3e4):
        x = to_bf16_bits(rng.standard_normal(64 * 16) * mag)
        g = oracle.calibrate_global_scale(x)
        scales, _ = _quantise_tensor(x, g)
        xv = bf16_bits_to_f64(x).reshape(-1, 16)
        assert scales.max() == 448.0                            # the block holding amax
        assert np.all(np.abs(xv).max(axis=1) / (6 * float(g)) <= 448.0 * (1 + 2**-4))


def test_calibration_bounds_the_error_where_unit_scale_clips():
    rng = np.random.default_rng(8)
    x = to_bf16_bits(rng.standard_normal(128 * 16) * 2e4)      # block maxima far above 6 * 448
    xv = bf16_bits_to_f64(x).reshape(-1, 16)
    bound = np.abs(xv).max(axis=1, keepdims=True) / 6 * (1 + 2**-4)
    _, deq = _quantise_tensor(x, oracle.calibrate_global_scale(x))
    assert np.all(np.abs(deq - xv) <= bound)                   # one E2M1 step of the block's scale
    _, deq1 = _quantise_tensor(x, 1.0)
    assert np.abs(deq1).max() <= 6 * 448                       # g = 1 clips at 2688 ...
    assert np.any(np.abs(deq1 - xv) > bound)                   # ... far outside that bound
