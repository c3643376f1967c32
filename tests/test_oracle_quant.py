"""Pins for the oracle's NVFP4 block quantisation, pool layout and append.

Closed forms (grid-valued blocks round-trip exactly), invariants (sign
symmetry, power-of-two equivariance), brute-force optimality of every code
and of the scale, and the byte ratio the page prints.
"""

import os

import numpy as np
import pytest
import torch

import oracle
from oracle_helpers import (GRID, bf16_bits_to_f64, codes_from_signed_grid, e4m3_values_all_positive,
                            e4m3_values_normal, grid_block, grid_rows, to_bf16_bits)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_byte_ratio_matches_page():
    g = read_golden("byte_ratio.txt")
    assert (g["nvfp4_data_bytes_per_block"] + g["nvfp4_scale_bytes_per_block"]) / g["fp8_bytes_per_block"] == g["ratio"]
    for P in (16, 32, 64, 128):
        nv = oracle.slab_bytes(oracle.DTYPE_NVFP4, P)
        f8 = oracle.slab_bytes(oracle.DTYPE_FP8, P)
        assert nv / f8 == g["ratio"]
        # per token per KV head: K and V, 128 values each
        assert nv == P * 2 * 128 * (g["nvfp4_data_bytes_per_block"] + g["nvfp4_scale_bytes_per_block"]) / 16


@pytest.mark.parametrize("seed", range(4))
def test_grid_valued_blocks_round_trip_exactly(seed):
    rng = np.random.default_rng(seed)
    codes_all, svals = e4m3_values_all_positive()
    for code_s, s in zip(codes_all, svals):
        x, e, _ = grid_block(rng, float(s))
        codes, sc = oracle.quantize_block16(to_bf16_bits(x))
        assert sc == code_s
        assert np.array_equal(codes, codes_from_signed_grid(e))


def _random_block(rng, scale=1.0):
    x = rng.standard_normal(16) * scale
    x[rng.random(16) < 0.1] *= 20.0
    return to_bf16_bits(x)


def test_sign_symmetry():
    rng = np.random.default_rng(1)
    for _ in range(2000):
        xb = _random_block(rng, 10.0 ** rng.uniform(-3, 2))
        c1, s1 = oracle.quantize_block16(xb)
        c2, s2 = oracle.quantize_block16(xb ^ np.uint16(0x8000))
        assert s1 == s2 and np.array_equal(c1 ^ 8, c2)


def test_power_of_two_equivariance():
    rng = np.random.default_rng(2)
    checked = 0
    for _ in range(2000):
        xb = _random_block(rng)
        x = bf16_bits_to_f64(xb)
        c1, s1 = oracle.quantize_block16(xb)
        k = int(rng.integers(-3, 4))
        c2, s2 = oracle.quantize_block16(to_bf16_bits(x * 2.0**k))
        v1, v2 = oracle.e4m3_value(s1), oracle.e4m3_value(s2)
        if v1 >= 2.0**-6 and v1 * 2.0**k >= 2.0**-6 and v1 * 2.0**k <= 448:   # both scales normal
            assert v2 == v1 * 2.0**k and np.array_equal(c1, c2)
            checked += 1
    assert checked > 1500


def test_every_code_and_scale_is_nearest():
    """Brute force: the scale is the nearest E4M3 value to amax/6 and each code
    the nearest grid value to x/scale (saturating at 6)."""
    rng = np.random.default_rng(3)
    _, svals = e4m3_values_all_positive()
    svals = np.concatenate([[0.0], svals])
    for _ in range(3000):
        xb = _random_block(rng, 10.0 ** rng.uniform(-4, 2))
        x = bf16_bits_to_f64(xb)
        codes, sc = oracle.quantize_block16(xb)
        sd = oracle.e4m3_value(sc)
        target = np.abs(x).max() / 6.0
        assert abs(sd - target) <= np.abs(svals - target).min()
        if sd == 0:
            assert np.all((codes & 7) == 0)
            continue
        xhat = np.array([oracle.e2m1_value(c) for c in codes]) * sd
        cand = np.concatenate([GRID, -GRID]) * sd
        for i in range(16):
            assert np.sign(xhat[i]) in (0.0, np.sign(x[i]))
            assert abs(xhat[i] - x[i]) <= np.abs(cand - x[i]).min() + 0.0
            if abs(x[i]) <= 6 * sd:
                assert abs(xhat[i] - x[i]) <= sd  # at most half the widest grid gap (2) times the scale


def test_zero_and_tiny_blocks():
    z = np.zeros(16, dtype=np.uint16)
    codes, sc = oracle.quantize_block16(z)
    assert sc == 0 and not codes.any()
    nz = np.full(16, 0x8000, dtype=np.uint16)  # -0.0
    codes, sc = oracle.quantize_block16(nz)
    assert sc == 0 and np.all(codes == 8)
    # amax/6 below half of the smallest E4M3 subnormal (2^-9) rounds the scale to 0
    tiny = to_bf16_bits(np.array([2.0**-12, -2.0**-12] * 8))
    codes, sc = oracle.quantize_block16(tiny)
    assert sc == 0 and np.array_equal(codes, np.array([0, 8] * 8, dtype=np.uint8))


def test_non_finite_input_rejected():
    with pytest.raises(ValueError):
        oracle.quantize_block16(np.array([0x7F80] + [0] * 15, dtype=np.uint16))


def _code_off(name, row):
    """The cache's documented layout: a slab is P/16 groups of 16 tokens, each
    K codes [16][64] | K scales [16][8] | V codes [16][64] | V scales [8][16]."""
    grp, r = divmod(row, 16)
    return grp * 2304 + (0 if name == "k" else 1152) + r * 64


def _scale_index(name, row, blk):
    grp, r = divmod(row, 16)
    if name == "k":
        return grp * 2304 + 1024 + r * 8 + blk
    return grp * 2304 + 2176 + blk * 16 + r


@pytest.mark.parametrize("P", [16, 64, 128])
def test_append_places_rows_at_documented_offsets(P):
    rng = np.random.default_rng(4)
    Hkv, T, num_pages = 3, 37, 9
    pool = oracle.OraclePool(num_pages, P, Hkv, fill=0xAB)
    k = grid_rows(rng, T * Hkv).reshape(T, Hkv, 128)
    v = grid_rows(rng, T * Hkv).reshape(T, Hkv, 128)
    slots = rng.permutation(num_pages * P)[:T].astype(np.int64)
    slots[5] = -1  # skipped
    oracle.quantize_append(pool, to_bf16_bits(k), to_bf16_bits(v), slots)
    touched = np.zeros((num_pages, P), dtype=bool)
    for t in range(T):
        if slots[t] < 0:
            continue
        page, row = divmod(int(slots[t]), P)
        touched[page, row] = True
        for h in range(Hkv):
            slab = pool.data[page, h]
            for name, src in (("k", k[t, h]), ("v", v[t, h])):
                q = slab[_code_off(name, row): _code_off(name, row) + 64]
                s = [slab[_scale_index(name, row, j)] for j in range(8)]
                vals = np.empty(128)
                for d in range(128):
                    code = (q[d // 2] >> (4 * (d % 2))) & 15
                    vals[d] = oracle.e2m1_value(int(code)) * oracle.e4m3_value(int(s[d // 16]))
                assert np.array_equal(vals, src)
    # untouched rows keep the fill byte
    for page in range(num_pages):
        for row in range(P):
            if touched[page, row]:
                continue
            for h in range(Hkv):
                slab = pool.data[page, h]
                for name in ("k", "v"):
                    assert np.all(slab[_code_off(name, row): _code_off(name, row) + 64] == 0xAB)
                    assert all(slab[_scale_index(name, row, j)] == 0xAB for j in range(8))


def test_append_rejects_out_of_range_slot():
    pool = oracle.OraclePool(2, 16, 1)
    k = np.zeros((1, 128), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.quantize_append(pool, k, k, np.array([32], dtype=np.int64))


def test_fp8_append_matches_torch_cast():
    rng = np.random.default_rng(5)
    P, Hkv, T = 16, 2, 20
    pool = oracle.OraclePool(4, P, Hkv, dtype=oracle.DTYPE_FP8)
    x = rng.standard_normal((T, Hkv, 128)) * 30
    k, v = to_bf16_bits(x), to_bf16_bits(-x * 0.5)
    slots = np.arange(T, dtype=np.int64) * 3 % (4 * P)
    oracle.quantize_append(pool, k, v, slots)
    for name, src in (("k", k), ("v", v)):
        ref = torch.from_numpy(bf16_bits_to_f64(src).astype(np.float32)).to(torch.float8_e4m3fn)
        ref = ref.view(torch.uint8).numpy()
        for t in range(T):
            page, row = divmod(int(slots[t]), P)
            for h in range(Hkv):
                grp, r = divmod(row, 16)
                base = grp * 4096 + (0 if name == "k" else 2048) + r * 128
                got = pool.data[page, h, base: base + 128]
                assert np.array_equal(got, ref[t, h])
