"""Small helpers for the oracle tests: BF16 bit conversion and grid-valued data.

A "grid-valued" block has every element equal to e_i * s with e_i on the
E2M1 grid and one element of magnitude exactly 6 * s, where s is an E4M3
value: then amax / 6 = s exactly, and quantising the block must return s and
the e_i unchanged (a closed form that needs no oracle).
"""

import numpy as np
import torch

GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def to_bf16_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def e4m3_values_normal():
    """Positive normal E4M3 values (exponent field 1..15, excluding NaN)."""
    codes = torch.arange(8, 0x7F, dtype=torch.uint8)
    return codes.numpy(), codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def e4m3_values_all_positive():
    codes = torch.arange(1, 0x7F, dtype=torch.uint8)
    return codes.numpy(), codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def grid_block(rng: np.random.Generator, s: float):
    """Returns (x[16] float64, e[16] signed grid values, index of the +-6 element)."""
    e = rng.choice(GRID, size=16) * rng.choice([-1.0, 1.0], size=16)
    j = int(rng.integers(16))
    e[j] = 6.0 * rng.choice([-1.0, 1.0])
    return e * s, e, j


def grid_rows(rng: np.random.Generator, n_rows: int, scale_choices=None) -> np.ndarray:
    """[n_rows][128] float64 rows made of 8 grid-valued blocks each."""
    if scale_choices is None:
        # scales in [2^-4, 8] keep every product comfortably inside BF16/FP16
        scale_choices = np.array([2.0**k * (1 + m / 8) for k in range(-4, 3) for m in range(8)])
    rows = np.empty((n_rows, 128))
    for r in range(n_rows):
        for b in range(8):
            x, _, _ = grid_block(rng, float(rng.choice(scale_choices)))
            rows[r, b * 16:(b + 1) * 16] = x
    return rows


def codes_from_signed_grid(e: np.ndarray) -> np.ndarray:
    """Signed grid values -> E2M1 codes (sign bit 3), -0 mapped to code 8."""
    mag = np.searchsorted(GRID, np.abs(e))
    assert np.array_equal(GRID[mag], np.abs(e))
    return np.where(np.signbit(e), mag | 8, mag).astype(np.uint8)
