"""Pins for the FP32 tensor scale g in the oracle's quantise / dequantise path.

NVFP4 stores code = E2M1(x / (s g)) with s = E4M3(amax / (6 g)), and reads
back e2m1 * e4m3 * g; the FP8 comparison cache stores E4M3(x / g) and reads
back e4m3 * g.  So (closed forms, no oracle needed for the expected values):
  * a power-of-two g changes no stored byte when the inputs are scaled by g,
    and the dequantised rows are the scaled inputs exactly;
  * for any other g the stored bytes are still those of the unscaled inputs
    (the BF16 rounding of x g is far inside the rounding margins), and each
    dequantised value is the FP32 product e2m1 * e4m3 * g rounded once to
    BF16, computed here with numpy's FP32 multiply and torch's BF16 cast.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle_helpers import bf16_bits_to_f64, grid_block, to_bf16_bits

P, HKV, T = 16, 2, 20


def _grid_tokens(rng):
    """[T][HKV][128] grid-valued values e * s, and each element's block scale s."""
    scales = np.array([2.0**k * (1 + m / 8) for k in range(-4, 3) for m in range(8)])
    x = np.empty((T, HKV, 128))
    s = np.empty((T, HKV, 128))
    for t in range(T):
        for h in range(HKV):
            for b in range(8):
                sc = float(rng.choice(scales))
                xb, _, _ = grid_block(rng, sc)
                x[t, h, 16 * b:16 * b + 16] = xb
                s[t, h, 16 * b:16 * b + 16] = sc
    return x, s


def _fill(dtype, gk, gv, k, v, slots):
    pool = oracle.OraclePool(3, P, HKV, dtype=dtype, gk=gk, gv=gv)
    oracle.quantize_append(pool, to_bf16_bits(k), to_bf16_bits(v), slots)
    return pool


def _dequant(pool):
    bt = np.array([[0, 1]], dtype=np.int32)   # the tokens sit on pages 0 and 1, in order
    return oracle.prefix_dequant(pool, bt, np.array([T], dtype=np.int32), np.array([0, T], dtype=np.int32))


def _bf16_of_fp32_product(a, g):
    prod = np.float32(a).astype(np.float32) * np.float32(g)   # one FP32 rounding
    return torch.from_numpy(np.ascontiguousarray(prod, dtype=np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


SLOTS = np.arange(T, dtype=np.int64)


@pytest.mark.parametrize("gk,gv", [(0.25, 8.0), (2.0, 0.5)])
def test_power_of_two_tensor_scale_is_lossless_and_changes_no_byte(gk, gv):
    rng = np.random.default_rng(int(gk * 16 + gv))
    k, _ = _grid_tokens(rng)
    v, _ = _grid_tokens(rng)
    unit = _fill(oracle.DTYPE_NVFP4, 1.0, 1.0, k, v, SLOTS)
    scaled = _fill(oracle.DTYPE_NVFP4, gk, gv, k * gk, v * gv, SLOTS)
    assert np.array_equal(unit.data, scaled.data)
    kw, vw = _dequant(scaled)
    assert np.array_equal(kw, to_bf16_bits(k * gk))
    assert np.array_equal(vw, to_bf16_bits(v * gv))


@pytest.mark.parametrize("g", [0.3, 3.7])
def test_other_tensor_scales_round_the_fp32_product_once_to_bf16(g):
    rng = np.random.default_rng(int(g * 10))
    k, _ = _grid_tokens(rng)
    v, _ = _grid_tokens(rng)
    kq = bf16_bits_to_f64(to_bf16_bits(k * g))
    vq = bf16_bits_to_f64(to_bf16_bits(v * g))
    unit = _fill(oracle.DTYPE_NVFP4, 1.0, 1.0, k, v, SLOTS)
    scaled = _fill(oracle.DTYPE_NVFP4, g, g, kq, vq, SLOTS)
    assert np.array_equal(unit.data, scaled.data)   # same codes and block scales
    kw, vw = _dequant(scaled)
    assert np.array_equal(kw, _bf16_of_fp32_product(k, g))
    assert np.array_equal(vw, _bf16_of_fp32_product(v, g))
    assert not np.array_equal(kw, to_bf16_bits(k))   # g is not a no-op


@pytest.mark.parametrize("g", [0.5, 0.3])
def test_fp8_tensor_scale(g):
    rng = np.random.default_rng(int(g * 100))
    codes = rng.integers(0, 0x7F, size=(2, T, HKV, 128)).astype(np.uint8)   # finite E4M3 codes
    codes |= (rng.integers(0, 2, size=codes.shape).astype(np.uint8) << 7)   # random signs
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    k, v = vals[0], vals[1]
    kq = bf16_bits_to_f64(to_bf16_bits(k * g))
    vq = bf16_bits_to_f64(to_bf16_bits(v * g))
    unit = _fill(oracle.DTYPE_FP8, 1.0, 1.0, k, v, SLOTS)
    scaled = _fill(oracle.DTYPE_FP8, g, g, kq, vq, SLOTS)
    assert np.array_equal(unit.data, scaled.data)   # E4M3(x g / g) = the code
    kw, vw = _dequant(scaled)
    assert np.array_equal(kw, _bf16_of_fp32_product(k, g))
    assert np.array_equal(vw, _bf16_of_fp32_product(v, g))
