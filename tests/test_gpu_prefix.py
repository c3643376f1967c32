"""GPU parity of prefix dequant: the BF16 workspace must equal the oracle's bit
for bit (ragged prefixes, shared pages, every page size, FP8 and tensor scales)."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import bits, fill_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import nvfp4_quantised_paged_gb300 as mod
    return mod


def _prefix_both(m, w, cache, pool, lens):
    pl = torch.tensor(lens, dtype=torch.int32)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(pl, 0)
    total = int(cu[-1])
    bt = w.block_table[:len(lens)].contiguous()
    kw, vw = m.prefix_dequant(cache, bt.cuda(), pl.cuda(), cu.cuda(), total)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    rk, rv = oracle.prefix_dequant(pool, bt.numpy(), pl.numpy(), cu.numpy())
    return bits(kw), bits(vw), rk, rv


@pytest.mark.parametrize("P", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", [0, 1])
def test_prefix_dequant_bit_exact(m, P, dtype):
    lens = [300, 1, 0, 1000, 64]
    w = workloads.make_decode("x", 40 + P, lens, 8, 2, P, recipe=workloads.ValueRecipe(outlier_p=0.01))
    cache, pool = fill_both(w, m, dtype=dtype)
    gk, gv, rk, rv = _prefix_both(m, w, cache, pool, [300, 1, 0, 999, 64])
    assert np.array_equal(gk, rk) and np.array_equal(gv, rv)


def test_prefix_dequant_with_tensor_scales(m):
    w = workloads.make_decode("y", 50, [500, 70], 8, 2, 64)
    for dtype in (0, 1):
        cache, pool = fill_both(w, m, dtype=dtype, gk=0.3, gv=1.7)
        gk, gv, rk, rv = _prefix_both(m, w, cache, pool, [500, 70])
        assert np.array_equal(gk, rk) and np.array_equal(gv, rv)


def test_agent_mix_extend_path(m):
    """Scaled-down agent mix: shared 3,200-token prefix, extends dequantise their
    prefixes and append a 512-token chunk, then decode sees the chunk."""
    mix = workloads.agent_mix(num_decode=4, num_extend=3)
    w = mix.decode
    cache, pool = fill_both(w, m)
    rows = mix.extend_rows()
    lens = [mix.extend_prefix_lens[i] for i in range(len(rows))]
    pl = torch.tensor(lens, dtype=torch.int32)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(pl, 0)
    bt = w.block_table[rows].contiguous()
    kw, vw = m.prefix_dequant(cache, bt.cuda(), pl.cuda(), cu.cuda(), int(cu[-1]))
    rk, rv = oracle.prefix_dequant(pool, bt.numpy(), pl.numpy(), cu.numpy())
    torch.cuda.synchronize()
    assert np.array_equal(bits(kw), rk) and np.array_equal(bits(vw), rv)
    for r in range(len(rows)):
        k, v = mix.chunk_kv(r, "cuda")
        slots = mix.chunk_slots(r)
        m.quantize_append(cache, k, v, slots.cuda())
        oracle.quantize_append(pool, bits(k), bits(v), slots.numpy())
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    assert np.array_equal(cache.pool.cpu().numpy(), pool.data)
