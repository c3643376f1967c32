"""Pins for the FP32 tensor scale g in the oracle's quantise / dequantise path,
against exact rational rounding (tests/exact_rounding.py, fractions.Fraction).

NVFP4 stores code = E2M1(x / (s g)) with s = E4M3(amax / (6 g)), each the
nearest-even rounding of the exact quotient, and its BF16 workspace holds
e2m1 * e4m3 * g rounded once to BF16; the FP8 comparison cache stores
E4M3(x / g) and reads back BF16(e4m3 * g).  The inputs sit at and next to
every rounding midpoint of the decision (the BF16 values nearest to
midpoint * divisor), for tensor scales that are not powers of two -- among
them scales found by search where forming the quotient in FP32 gives another
code than exact rounding, and where rounding the product to FP32 before BF16
gives another BF16 value, so that either shortcut fails these tests.
"""

from fractions import Fraction as Fr

import numpy as np
import pytest

import oracle
import probes
from exact_rounding import E2M1, E4M3, bf16_rne_bits, bf16_value, rne_code
from oracle_helpers import bf16_bits_to_f64, grid_block, to_bf16_bits
from probes import E2M1_MIDS, G_SET, f32

P, HKV, T = 16, 2, 20

FP32_SCALE_TRAPS = probes.scale_traps()
FP32_PRODUCT_TRAPS = probes.product_traps()


def test_searches_found_traps():
    assert len(FP32_SCALE_TRAPS) >= 2 and len(FP32_PRODUCT_TRAPS) >= 2


@pytest.mark.parametrize("g", G_SET + [t[0] for t in FP32_SCALE_TRAPS])
def test_scale_is_the_exact_rounding_at_every_midpoint(g):
    blocks = probes.scale_probe_blocks(g)
    assert len(blocks) > 500
    for x in blocks:
        _, s = oracle.quantize_block16(x, g)
        assert s == rne_code(bf16_value(int(x[0]) & 0x7FFF) / (6 * Fr(g)), E4M3), (g, hex(int(x[0])))


def test_fp32_traps_are_decided_exactly():
    for g, a_bits, exact in FP32_SCALE_TRAPS:
        _, s = oracle.quantize_block16(probes.block(a_bits), g)
        assert s == exact != probes.fp32_scale_code(a_bits, g)


@pytest.mark.parametrize("g", G_SET[:6] + [t[0] for t in FP32_SCALE_TRAPS[:2]])
def test_codes_are_the_exact_rounding_at_every_midpoint(g):
    G = Fr(g)
    blocks, scales = probes.code_probe_blocks(g)
    n_ties = n = 0
    for x, sc in zip(blocks, scales):
        codes, s = oracle.quantize_block16(x, g)
        assert s == sc
        den = E4M3[sc] * G
        for j in range(1, 16):
            if x[j] == 0 and j > 1:
                continue
            q = bf16_value(int(x[j]) & 0x7FFF) / den
            want = rne_code(q, E2M1) | (8 if x[j] & 0x8000 else 0)
            assert codes[j] == want, (g, sc, hex(int(x[j])))
            n += 1
            n_ties += int(q in E2M1_MIDS)
    assert n > 300
    if g in (1.5, 0.75):
        assert n_ties > 0        # exact ties occur (BF16 x equal to midpoint * s * g)


@pytest.mark.parametrize("g", [f32(0.3), 1.5, f32(2.0**-110 * 1.37), f32(2.0**90 * 1.9)])
def test_fp8_codes_are_the_exact_rounding_at_every_midpoint(g):
    xs = probes.fp8_probe_values(g)
    k = probes.rows_of(xs)
    rows = k.shape[0]
    pool = oracle.OraclePool(-(-rows // 16), 16, 1, dtype=oracle.DTYPE_FP8, gk=g, gv=g)
    oracle.quantize_append(pool, k, k, np.arange(rows, dtype=np.int64))
    for i, b in enumerate(xs):
        r, d = divmod(i, 128)
        got = pool.data[r // 16, 0, (r % 16) * 128 + d]      # P = 16: K codes [16][128] of each page
        want = rne_code(bf16_value(int(b) & 0x7FFF) / Fr(g), E4M3) | (0x80 if b & 0x8000 else 0)
        assert got == want, (g, hex(int(b)))


# ----------------------------------------------------------------- dequant: BF16 of the exact product


def _dequant_all(pool, rows):
    pages = np.arange(pool.num_pages, dtype=np.int32)[None]
    return oracle.prefix_dequant(pool, pages, np.array([rows], np.int32), np.array([0, rows], np.int32))


def _signed_zero_bits(c, s):
    """Sign of the exact product e2m1 * e4m3 * g when it is zero (IEEE: the XOR of the signs)."""
    return 0x8000 if bool(c & 8) != bool(s & 0x80) else 0


@pytest.mark.parametrize("g", [1.0, 0.25, f32(0.3), f32(3.7), f32(1.0 / 2688), f32(2.0**-120 * 1.5),
                               f32(2.0**-126), f32(2.0**100 * 1.7), f32(3.0e38)])
def test_nvfp4_dequant_is_the_exact_product_rounded_once(g):
    _check_nvfp4_dequant(g)


@pytest.mark.parametrize("i", range(3))
def test_nvfp4_dequant_at_fp32_product_traps(i):
    if i >= len(FP32_PRODUCT_TRAPS):
        pytest.skip("fewer traps found")
    _check_nvfp4_dequant(FP32_PRODUCT_TRAPS[i], want_double_rounding_cases=True)


def _check_nvfp4_dequant(g, want_double_rounding_cases=False):
    pairs = probes.all_products()
    pool, rows = probes.crafted_pool(oracle.DTYPE_NVFP4, g)
    kw, vw = _dequant_all(pool, rows)
    got_k = kw.reshape(-1)[:len(pairs)]
    got_v = vw.reshape(-1)[:len(pairs)]
    G = Fr(g)
    n_double = 0
    for i, (c, s) in enumerate(pairs):
        e = E2M1[c & 7] * (-1 if c & 8 else 1)
        sv = E4M3[s & 0x7F] * (-1 if s & 0x80 else 1)
        exact = e * sv * G
        want = bf16_rne_bits(exact) if exact != 0 else _signed_zero_bits(c, s)
        assert got_k[i] == want and got_v[i] == want, (g, c, s, hex(int(got_k[i])), hex(want))
        if want_double_rounding_cases and exact != 0:
            fp32 = np.float32(float(e * sv)) * np.float32(g)    # an IEEE FP32 product: one rounding
            n_double += int(bf16_rne_bits(Fr(float(fp32))) != want)
    if want_double_rounding_cases:
        assert n_double > 0


@pytest.mark.parametrize("g", [1.0, f32(0.3), f32(2.0**-120 * 1.5), f32(3.0e38)] + FP32_PRODUCT_TRAPS[:1])
def test_fp8_dequant_is_the_exact_product_rounded_once(g):
    codes = list(range(0, 127)) + list(range(128, 255))
    pool, rows = probes.crafted_pool(oracle.DTYPE_FP8, g)
    kw, vw = _dequant_all(pool, rows)
    G = Fr(g)
    for i, c in enumerate(codes):
        exact = E4M3[c & 0x7F] * (-1 if c & 0x80 else 1) * G
        want = bf16_rne_bits(exact) if exact != 0 else (0x8000 if c & 0x80 else 0)
        assert kw.reshape(-1)[i] == want and vw.reshape(-1)[i] == want, (g, c)


# ----------------------------------------------------------------- closed forms


def _grid_tokens(rng):
    """[T][HKV][128] grid-valued values e * s."""
    scales = np.array([2.0**k * (1 + m / 8) for k in range(-4, 3) for m in range(8)])
    x = np.empty((T, HKV, 128))
    for t in range(T):
        for h in range(HKV):
            for b in range(8):
                xb, _, _ = grid_block(rng, float(rng.choice(scales)))
                x[t, h, 16 * b:16 * b + 16] = xb
    return x


def _fill(dtype, gk, gv, k, v, slots):
    pool = oracle.OraclePool(3, P, HKV, dtype=dtype, gk=gk, gv=gv)
    oracle.quantize_append(pool, to_bf16_bits(k), to_bf16_bits(v), slots)
    return pool


def _dequant(pool):
    bt = np.array([[0, 1]], dtype=np.int32)   # the tokens sit on pages 0 and 1, in order
    return oracle.prefix_dequant(pool, bt, np.array([T], dtype=np.int32), np.array([0, T], dtype=np.int32))


SLOTS = np.arange(T, dtype=np.int64)


@pytest.mark.parametrize("gk,gv", [(0.25, 8.0), (2.0, 0.5)])
def test_power_of_two_tensor_scale_is_lossless_and_changes_no_byte(gk, gv):
    rng = np.random.default_rng(int(gk * 16 + gv))
    k = _grid_tokens(rng)
    v = _grid_tokens(rng)
    unit = _fill(oracle.DTYPE_NVFP4, 1.0, 1.0, k, v, SLOTS)
    scaled = _fill(oracle.DTYPE_NVFP4, gk, gv, k * gk, v * gv, SLOTS)
    assert np.array_equal(unit.data, scaled.data)
    kw, vw = _dequant(scaled)
    assert np.array_equal(kw, to_bf16_bits(k * gk))
    assert np.array_equal(vw, to_bf16_bits(v * gv))


@pytest.mark.parametrize("g", [0.3, 3.7])
def test_other_tensor_scales_keep_the_codes_of_scaled_grid_values(g):
    """BF16(x g) of grid-valued x lies within 2^-9 of x g, far inside every
    rounding margin: the stored codes and scales are those of x at g = 1."""
    g = f32(g)
    rng = np.random.default_rng(int(g * 10))
    k = _grid_tokens(rng)
    v = _grid_tokens(rng)
    kq = bf16_bits_to_f64(to_bf16_bits(k * g))
    vq = bf16_bits_to_f64(to_bf16_bits(v * g))
    unit = _fill(oracle.DTYPE_NVFP4, 1.0, 1.0, k, v, SLOTS)
    scaled = _fill(oracle.DTYPE_NVFP4, g, g, kq, vq, SLOTS)
    assert np.array_equal(unit.data, scaled.data)


def test_invalid_tensor_scales_are_rejected():
    x = np.zeros(16, dtype=np.uint16)
    for g in (0.0, -1.0, float("inf"), float("nan"), 1e-40):
        with pytest.raises(ValueError):
            oracle.quantize_block16(x, g)
