"""GPU parity at tensor scales g != 1, bit for bit against the oracle (itself
pinned to exact rational rounding): quantise-append of inputs placed at and next
to every rounding midpoint of the scale and code decisions -- for scales that are
not powers of two, the smallest normal and near-largest FP32 scales, and scales
where an FP32 quotient would decide differently -- and prefix dequant of every
(E2M1 code, E4M3 scale) pair and every FP8 code, including scales where rounding
the product to FP32 before BF16 would differ."""

import numpy as np
import pytest
import torch

import oracle
import probes
from gpu_common import bits

pytestmark = pytest.mark.gpu

SCALE_TRAPS = [t[0] for t in probes.scale_traps()]
PRODUCT_TRAPS = probes.product_traps()


@pytest.fixture(scope="module")
def m():
    import nvfp4_quantised_paged_gb300 as mod
    return mod


def _bf16(u16):
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("g", probes.G_SET + SCALE_TRAPS)
def test_append_at_every_midpoint_matches_oracle(m, g):
    code_blocks, _ = probes.code_probe_blocks(g)
    blocks = np.concatenate([probes.scale_probe_blocks(g)] + ([code_blocks] if len(code_blocks) else []))
    k = probes.rows_of(blocks.reshape(-1))
    v = k ^ np.uint16(0x8000)
    T = k.shape[0]
    P = 16
    pages = -(-T // P)
    slots = torch.randperm(pages * P, generator=torch.Generator().manual_seed(7))[:T].to(torch.int64)
    for dtype, (kk, vv) in ((0, (k, v)), (1, (probes.rows_of(probes.fp8_probe_values(g)),) * 2)):
        n = kk.shape[0]
        cache = m.PagedCache(pages, P, 1, dtype=dtype, k_global_scale=g, v_global_scale=g)
        m.quantize_append(cache, _bf16(kk).cuda(), _bf16(vv).cuda(), slots[:n].cuda())
        pool = oracle.OraclePool(pages, P, 1, dtype=dtype, gk=g, gv=g)
        oracle.quantize_append(pool, kk, vv, slots[:n].numpy())
        torch.cuda.synchronize()
        assert m.check_device_errors() == 0
        assert np.array_equal(cache.pool.cpu().numpy(), pool.data), "dtype %d g %r" % (dtype, g)


@pytest.mark.parametrize("g", [0.25, probes.f32(0.3), probes.f32(3.7), probes.f32(2.0**-120 * 1.5),
                               probes.f32(2.0**-126), probes.f32(2.0**100 * 1.7), probes.f32(3.0e38)] + PRODUCT_TRAPS)
@pytest.mark.parametrize("dtype", [0, 1])
def test_prefix_dequant_of_every_product_matches_oracle(m, g, dtype):
    pool, rows = probes.crafted_pool(dtype, g)
    cache = m.PagedCache(pool.num_pages, pool.page_size, 1, dtype=dtype, k_global_scale=g, v_global_scale=g,
                         pool=torch.from_numpy(pool.data.copy()).cuda())
    bt = np.arange(pool.num_pages, dtype=np.int32)[None]
    pl, cu = np.array([rows], np.int32), np.array([0, rows], np.int32)
    kw, vw = m.prefix_dequant(cache, torch.from_numpy(bt).cuda(), torch.from_numpy(pl).cuda(),
                              torch.from_numpy(cu).cuda(), rows)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    rk, rv = oracle.prefix_dequant(pool, bt, pl, cu)
    assert np.array_equal(bits(kw), rk) and np.array_equal(bits(vw), rv)


def test_subnormal_tensor_scale_is_refused(m):
    cache = m.PagedCache(1, 16, 1, k_global_scale=1e-40)
    k = torch.zeros((1, 1, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.NVFP4KVError):
        m.quantize_append(cache, k, k, torch.zeros(1, dtype=torch.int64, device="cuda"))
