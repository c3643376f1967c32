"""The exact-rounding helpers the tensor-scale pins rely on, checked against
library routines and closed forms: torch's float32 -> bfloat16 cast (nearest
even, subnormals, overflow; a Fraction has no signed zero, so -0 is left to the callers) for bf16_rne_bits, torch's float8_e4m3fn decoding
for the E4M3 table, and the E2M1 tie cases written out by hand."""

from fractions import Fraction as Fr

import numpy as np
import torch

from exact_rounding import E2M1, E4M3, bf16_neighbours, bf16_rne_bits, bf16_value, rne_code


def test_bf16_rounding_matches_torch_cast():
    rng = np.random.default_rng(0)
    xs = (rng.standard_normal(4000) * 10.0 ** rng.integers(-44, 39, 4000)).astype(np.float32)
    xs = np.concatenate([xs, np.float32([3.3e38, 3.39e38, -3.4e38, 1e-40, -2e-45, 0.0])])
    want = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for x, w in zip(xs, want):
        if x == 0:
            continue    # a Fraction has no signed zero
        assert bf16_rne_bits(Fr(float(x))) == int(w), float(x)
    assert bf16_rne_bits(Fr(0)) == 0


def test_bf16_ties_go_to_even():
    assert bf16_rne_bits(Fr(1) + Fr(1, 256)) == 0x3F80              # 1 + half a step -> 1
    assert bf16_rne_bits(Fr(1) + Fr(3, 256)) == 0x3F82              # 1 + 1.5 steps -> 1 + 2 steps
    assert bf16_rne_bits(Fr(1) + Fr(1, 256) + Fr(1, 2**40)) == 0x3F81


def test_e4m3_table_matches_torch():
    want = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert [float(v) for v in E4M3] == list(want)


def test_e2m1_ties_and_saturation():
    cases = {Fr(1, 4): 0, Fr(3, 4): 2, Fr(5, 4): 2, Fr(7, 4): 4, Fr(5, 2): 4, Fr(7, 2): 6, Fr(5): 6, Fr(7): 7,
             Fr(1, 4) + Fr(1, 10**9): 1, Fr(0): 0}
    for q, c in cases.items():
        assert rne_code(q, E2M1) == c, q


def test_neighbours_bracket_the_target():
    for t in (Fr(1, 3), Fr(1000, 7), Fr(6) * Fr(1, 2688)):
        ns = [bf16_value(b) for b in bf16_neighbours(t, 1)]
        assert min(ns) < t < max(ns) and len(ns) >= 4
