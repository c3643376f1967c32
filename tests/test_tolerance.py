"""The attention tolerance of the GPU parity tests, on the CPU:
|got - ref| <= max(2e-2, half a BF16 step at |ref| + eta, plus eta), with
eta = (eps + 2^-16) spread + 2^-16 |ref|, and relative L2 <= 3e-3.  The bar
is exactly 2e-2 below |ref| = 8 while the oracle's spread is that of
well-behaved rows, it admits the BF16 rounding of any real, it grows with the
spread by eps, and it is reached and not exceeded."""

import numpy as np
import pytest
import torch

from gpu_common import EPS_BF16_P, EPS_FP16_P, FP32_REL, MAX_ABS, REL_L2, attention_bound, bf16_ulp, check_attention


def test_bf16_step():
    x = np.array([1.0, 1.5, 1.9999, 2.0, 0.5, 8.0, 15.9, -3.0, 2.0**-120])
    want = np.array([2**-7, 2**-7, 2**-7, 2**-6, 2**-8, 2**-4, 2**-4, 2**-6, 2.0**-127])
    assert np.array_equal(bf16_ulp(x), want)


def test_bar_is_2e2_below_8():
    ref = np.linspace(-7.9, 7.9, 20001)
    # spread 1 (values around the output at the scale of N(0,1) data)
    assert np.all(attention_bound(ref, np.ones_like(ref)) == MAX_ABS)
    # with BF16 probabilities 2e-2 holds too below 4 for that spread
    r4 = np.linspace(-3.9, 3.9, 999)
    assert np.all(attention_bound(r4, np.ones_like(r4), EPS_BF16_P) == MAX_ABS)
    # half a step at [8, 16) is 2^-5, beyond 2e-2: the bar is half a step + eta there
    r = np.array([8.0, 12.0, 15.9])
    eta = (EPS_FP16_P + FP32_REL) * 2.0 + FP32_REL * r
    assert np.allclose(attention_bound(r, np.full(3, 2.0)), 2.0**-5 + eta)


def test_bar_grows_with_spread():
    ref = np.zeros(3)
    s = np.array([10.0, 50.0, 200.0])
    want = np.maximum(MAX_ABS, 0.5 * bf16_ulp((EPS_BF16_P + FP32_REL) * s) + (EPS_BF16_P + FP32_REL) * s)
    assert np.array_equal(attention_bound(ref, s, EPS_BF16_P), want)
    assert attention_bound(ref, s)[0] == MAX_ABS            # 10 x 2^-11 < 2e-2


def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def test_rounding_to_bf16_passes_everywhere():
    rng = np.random.default_rng(3)
    ref = np.concatenate([rng.uniform(-64, 64, 4000), rng.uniform(-1, 1, 4000), [7.999, 8.0, 15.99, 31.9]])
    check_attention(_bf16(ref), ref, "rounded", spread=np.zeros_like(ref))   # the best a BF16 output can do


def test_bound_is_tight_per_element():
    z = np.zeros(1000)
    ref = np.full(1000, 0.5)
    got = ref.copy()
    got[7] += MAX_ABS * 0.99      # inside (and in BF16: 0.5 + 0.0198 rounds to 0.51953125, err 0.0195)
    check_attention(_bf16(got), ref, "inside", spread=z)
    got[7] = 0.5 + 0.03125        # exactly representable, beyond 2e-2
    with pytest.raises(AssertionError):
        check_attention(_bf16(got), ref, "beyond", spread=z)
    # in [4, 8) a BF16 step (2^-5 = 0.03125) is beyond the bar: 2e-2 holds there
    five = np.full(100, 5.0)
    one = five.copy()
    one[3] += 0.03125
    with pytest.raises(AssertionError):
        check_attention(_bf16(one), five, "one step at 5", spread=np.ones(100))
    # at 12 a step is 0.0625 and half a step 0.03125: the nearest BF16 passes, one step beyond fails
    big = np.full(100, 12.0)
    big[3] = 12.03
    check_attention(_bf16(big), big, "nearest BF16 to 12.03", spread=np.zeros(100))
    off = big.copy()
    off[3] = 12.0625 + 0.0625
    with pytest.raises(AssertionError):
        check_attention(_bf16(off), big, "one step beyond the nearest at 12", spread=np.ones(100))


def test_spread_widens_the_bar_by_eps():
    ref = np.full(100000, 0.25)
    got = ref.copy()
    got[2] += 0.04
    with pytest.raises(AssertionError):
        check_attention(_bf16(got), ref, "small spread", spread=np.ones(ref.size))
    check_attention(_bf16(got), ref, "spread 100 with BF16 probabilities", eps=EPS_BF16_P,
                    spread=np.full(ref.size, 100.0))


def test_two_rounded_outputs_get_a_full_step():
    ref = np.full(10, 12.0)
    got = ref.copy()
    got[2] += 0.0625
    with pytest.raises(AssertionError):
        check_attention(_bf16(got), ref + 0.001, "half step", spread=np.zeros(10))
    check_attention(_bf16(got), ref, "full step", spread=np.zeros(10), both_rounded=True)


def test_spread_is_required():
    with pytest.raises(TypeError):
        check_attention(_bf16([1.0]), np.ones(1), "no spread")


def test_relative_l2_bound():
    rng = np.random.default_rng(4)
    ref = rng.standard_normal(20000)
    small = ref + 1e-3 * rng.standard_normal(ref.size)      # rel-L2 about 1e-3 plus BF16 rounding
    check_attention(_bf16(small), ref, "small", spread=np.ones_like(ref))
    biased = ref * (1.0 + 2 * REL_L2)                        # every element within 2e-2, rel-L2 6e-3
    with pytest.raises(AssertionError):
        check_attention(_bf16(biased), ref, "biased", spread=np.ones_like(ref))


def test_non_finite_output_fails():
    with pytest.raises(AssertionError):
        check_attention(_bf16([0.0, float("nan")]), np.zeros(2), "nan", spread=np.zeros(2))
