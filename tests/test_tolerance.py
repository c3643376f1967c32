"""The attention tolerance of the GPU parity tests, on the CPU: per element
|got - ref| <= max(2e-2, one BF16 step at |ref|), relative L2 <= 3e-3.
The bound is reached and not exceeded, and the BF16 rounding of any real in
[8, 16) (up to half a step, 2^-5 > 2e-2) stays inside it."""

import numpy as np
import pytest
import torch

from gpu_common import MAX_ABS, REL_L2, bf16_ulp, check_attention


def test_bf16_step():
    x = np.array([1.0, 1.5, 1.9999, 2.0, 0.5, 8.0, 15.9, -3.0, 2.0**-120])
    want = np.array([2**-7, 2**-7, 2**-7, 2**-6, 2**-8, 2**-4, 2**-4, 2**-6, 2.0**-127])
    assert np.array_equal(bf16_ulp(x), want)


def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def test_rounding_to_bf16_passes_everywhere():
    rng = np.random.default_rng(3)
    ref = np.concatenate([rng.uniform(-16, 16, 4000), rng.uniform(-1, 1, 4000)])
    check_attention(_bf16(ref), ref, "rounded")   # the best a BF16 output can do


def test_bound_is_tight_per_element():
    ref = np.full(1000, 0.5)
    got = ref.copy()
    got[7] += MAX_ABS * 0.99      # inside (and in BF16: 0.5 + 0.0198 rounds to 0.51953125, err 0.0195)
    check_attention(_bf16(got), ref, "inside")
    got[7] = 0.5 + 0.03125        # exactly representable, beyond 2e-2
    with pytest.raises(AssertionError):
        check_attention(_bf16(got), ref, "beyond")
    big = np.full(100, 12.0)
    one = big.copy()
    one[3] += 0.0625                                          # one BF16 step at 12 is allowed there
    check_attention(_bf16(one), big, "one step at 12")
    two = big.copy()
    two[3] += 0.125
    with pytest.raises(AssertionError):
        check_attention(_bf16(two), big, "two steps at 12")


def test_relative_l2_bound():
    rng = np.random.default_rng(4)
    ref = rng.standard_normal(20000)
    small = ref + 1e-3 * rng.standard_normal(ref.size)      # rel-L2 about 1e-3 plus BF16 rounding
    check_attention(_bf16(small), ref, "small")
    biased = ref * (1.0 + 2 * REL_L2)                        # every element within 2e-2, rel-L2 6e-3
    with pytest.raises(AssertionError):
        check_attention(_bf16(biased), ref, "biased")


def test_non_finite_output_fails():
    with pytest.raises(AssertionError):
        check_attention(_bf16([0.0, float("nan")]), np.zeros(2), "nan")
