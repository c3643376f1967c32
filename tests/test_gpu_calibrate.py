"""Tensor-scale calibration on the GPU against the oracle: the scales
themselves bit for bit (plain, outlier, huge, tiny, Inf/NaN-carrying and
token-strided tensors, and the empty one), then a cache filled with the
calibrated scales -- its bytes bit-exact and its decode attention within
tolerance of the oracle run with the same scales -- on activations large
enough that a unit tensor scale would clip every block."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import bits, check_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import nvfp4_quantised_paged_gb300 as mod
    return mod


def _kv(T, Hkv, seed, scale=1.0, recipe=None):
    recipe = recipe or workloads.ValueRecipe()
    k = workloads.draw_kv(T, Hkv, seed, 0, "cuda", recipe, 0)
    v = workloads.draw_kv(T, Hkv, seed, 0, "cuda", recipe, 1)
    if scale != 1.0:
        k, v = (k.float() * scale).to(torch.bfloat16), (v.float() * scale).to(torch.bfloat16)
    return k, v


def _check_scales(m, k, v, Hkv):
    got = m.calibrate_global_scales(k, v, Hkv).cpu().numpy()
    ref = np.array([oracle.calibrate_global_scale(bits(k)), oracle.calibrate_global_scale(bits(v))],
                   dtype=np.float32)
    assert got.dtype == np.float32 and np.array_equal(got.view(np.uint32), ref.view(np.uint32)), (got, ref)
    return got


@pytest.mark.parametrize("scale", [1.0, 3e4, 1e-30])
def test_scales_match_oracle(m, scale):
    k, v = _kv(5000, 8, 11, scale, workloads.ValueRecipe(outlier_p=0.002, zero_block_p=0.01))
    _check_scales(m, k, v, 8)


def test_scales_ignore_inf_and_nan_and_follow_strides(m):
    k, v = _kv(777, 4, 12)
    k[5, 1, 7] = float("inf")
    k[9, 0, 0] = float("nan")
    v[700, 3, 127] = -float("inf")
    _check_scales(m, k, v, 4)
    wide = torch.zeros((777, 3 * 4 * 128), dtype=torch.bfloat16, device="cuda")   # a fused QKV-like buffer
    wide[:, 512:1024] = k.reshape(777, 512)
    wide[:, 1024:1536] = v.reshape(777, 512)
    wide[:, :512] = 1e6                                                            # not part of K or V
    got = m.calibrate_global_scales(wide[:, 512:1024], wide[:, 1024:1536], 4).cpu().numpy()
    ref = _check_scales(m, k, v, 4)
    assert np.array_equal(got, ref)


def test_zero_and_empty_tensors_give_unit_scales(m):
    z = torch.zeros((10, 2, 128), dtype=torch.bfloat16, device="cuda")
    assert m.calibrate_global_scales(z, z, 2).tolist() == [1.0, 1.0]
    e = torch.zeros((0, 2, 128), dtype=torch.bfloat16, device="cuda")
    assert m.calibrate_global_scales(e, e, 2).tolist() == [1.0, 1.0]


def test_calibrated_cache_and_decode_match_oracle(m):
    w = workloads.make_decode("calibrated", 21, [700, 1500, 64, 333], 32, 8, 64)
    ks, vs = [], []
    for b in range(w.batch):
        k, v = w.seq_kv(b, "cuda")
        ks.append((k.float() * 2e4).to(torch.bfloat16))   # block maxima far above 6 * 448
        vs.append((v.float() * 5e3).to(torch.bfloat16))
    g = _check_scales(m, torch.cat(ks), torch.cat(vs), 8)
    gk, gv = float(g[0]), float(g[1])
    assert gk > 1.0 and gv > 1.0
    cache = m.PagedCache(w.num_pages, w.page_size, w.num_kv_heads, k_global_scale=gk, v_global_scale=gv)
    pool = oracle.OraclePool(w.num_pages, w.page_size, w.num_kv_heads, gk=gk, gv=gv)
    for b in range(w.batch):
        slots = w.slots(b)
        m.quantize_append(cache, ks[b], vs[b], slots.cuda())
        oracle.quantize_append(pool, bits(ks[b]), bits(vs[b]), slots.numpy())
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    assert np.array_equal(cache.pool.cpu().numpy(), pool.data)
    q = (w.q("cuda").float() / 2e4).to(torch.bfloat16)   # keeps the scores O(1)
    out = m.paged_decode_attention(cache, q, w.block_table.cuda(), w.seq_lens.cuda(), w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    ref, spread = oracle.decode_attention(pool, bits(q), w.block_table.numpy(), w.seq_lens.numpy(), w.sm_scale,
                                          spread=True)
    check_attention(out / 5e3, ref / 5e3, "calibrated decode (in units of the V scale-up)", spread=spread / 5e3)
