"""Host checks of the arithmetic shortcuts the CUDA quantiser takes, against
the definitions the oracle follows (section A3 / Fig. 1: the block scale is
E4M3 of amax / (6 g), the quotient formed in FP32).

The unit-scale path of the GPU quantiser multiplies amax by fl32(1/6) instead
of dividing by 6.  Their FP32 results differ for some amax, but the E4M3
scale they round to must not: this is checked here over every finite
non-negative BF16 value, which is every amax a block can have.  It forms the
element quotients as a product by an approximate reciprocal rounded to FP16;
that the codes are those of the quotients is checked over every BF16 value,
every E4M3 scale and every reciprocal within two units of the correct one."""

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


def _e4m3_positive_values():
    return np.array([oracle.e4m3_value(c) for c in range(1, 127)], dtype=np.float32)


def test_fp16_rounded_reciprocal_product_gives_the_quotients_e2m1_code():
    """The unit-scale GPU path forms y = fl32(x * r) with r the hardware's
    approximate reciprocal of the block scale, rounds y to FP16 and converts
    that to E2M1 (infinity saturating to 6).  For every finite non-negative
    BF16 x, every positive E4M3 scale and every r within two units in the last
    place of fl32(1 / scale), the code must be the one of the quotient."""
    x = _all_bf16_magnitudes()
    n_crossed = 0
    for sd in _e4m3_positive_values():
        want = oracle.e2m1_encode_quotients(x, sd)
        r0 = np.array([np.float32(1.0) / sd], dtype=np.float32)
        for k in (-2, -1, 0, 1, 2):
            r = (r0.view(np.int32) + np.int32(k)).view(np.float32)[0]
            with np.errstate(over="ignore"):   # products beyond FP32 / FP16: infinity, which saturates
                y = (x * r).astype(np.float32)
                h = y.astype(np.float16).astype(np.float32)
            h = np.where(np.isinf(h), np.float32(65504.0), h)
            got = oracle.e2m1_encode_quotients(h, np.float32(1.0))
            assert np.array_equal(got, want), (float(sd), k)
            # the FP32 product alone (without the FP16 rounding) would round some exact midpoints the wrong way
            n_crossed += int((oracle.e2m1_encode_quotients(y, np.float32(1.0)) != want).sum())
    assert n_crossed > 0
