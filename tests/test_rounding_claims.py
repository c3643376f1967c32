"""Host checks of the arithmetic shortcuts the CUDA quantiser takes, against
the definitions the oracle follows (section A3 / Fig. 1: the block scale is
E4M3 of amax / (6 g), the quotient formed in FP32).

The unit-scale path of the GPU quantiser multiplies amax by fl32(1/6) instead
of dividing by 6.  Their FP32 results differ for some amax, but the E4M3
scale they round to must not: this is checked here over every finite
non-negative BF16 value, which is every amax a block can have."""

import numpy as np

import oracle


def _all_bf16_magnitudes():
    bits = np.arange(0, 0x7F80, dtype=np.uint32)  # exponent field < 255: zero, subnormals, normals
    return (bits << 16).view(np.float32)


def test_one_sixth_product_gives_the_quotients_e4m3_scale():
    amax = _all_bf16_magnitudes()
    by_div = (amax / np.float32(6.0)).astype(np.float32)
    one_sixth = np.float32(1.0) / np.float32(6.0)
    by_mul = (amax * one_sixth).astype(np.float32)
    assert (by_div != by_mul).any()  # the shortcut is not exact in FP32 ...
    e_div = oracle.e4m3_encode_many(by_div.astype(np.float64))
    e_mul = oracle.e4m3_encode_many(by_mul.astype(np.float64))
    assert np.array_equal(e_div, e_mul)  # ... but the scale decision is


def test_one_sixth_constant_is_the_rounded_reciprocal():
    # the kernel's literal must be fl32(1/6)
    assert np.float32(0.16666667163372039794921875) == np.float32(1.0) / np.float32(6.0)
    assert float(np.float32(1.0) / np.float32(6.0)) == 0.16666667163372039794921875
