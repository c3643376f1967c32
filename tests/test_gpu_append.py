"""GPU parity of quantise-append: packed codes and scales must equal the
oracle's bit for bit, over every BF16 value against every E4M3 scale, over
seeded workloads with outliers and all-zero blocks, and for every page size."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import nvfp4_quantised_paged_gb300 as mod
    return mod


def _append_both(m, k, v, slots, num_pages, P, Hkv, dtype=0, gk=1.0, gv=1.0):
    cache = m.PagedCache(num_pages, P, Hkv, dtype=dtype, k_global_scale=gk, v_global_scale=gv)
    m.quantize_append(cache, k.cuda(), v.cuda(), slots.cuda())
    pool = oracle.OraclePool(num_pages, P, Hkv, dtype=dtype, gk=gk, gv=gv)
    oracle.quantize_append(pool, bits(k), bits(v), slots.numpy())
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    return cache.pool.cpu().numpy(), pool.data


def test_every_bf16_value_against_every_scale():
    """Each block holds 6*s (so its scale is exactly s) and 15 BF16 values of
    magnitude <= 6*s; together the blocks cover every BF16 magnitude below
    6*s, both signs, for each of the 126 positive E4M3 scales s."""
    import nvfp4_quantised_paged_gb300 as m
    allbits = np.arange(1 << 15, dtype=np.uint32).astype(np.uint16)   # non-negative BF16 patterns
    mags = oracle.bf16_to_f64(allbits)
    finite = np.isfinite(mags)
    allbits, mags = allbits[finite], mags[finite]
    codes = torch.arange(1, 0x7F, dtype=torch.uint8)
    scales = codes.view(torch.float8_e4m3fn).double().numpy()
    blocks = []
    for s in scales:
        top = 6.0 * s
        top_bits = torch.tensor([top], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        sel = allbits[mags <= top]
        vals = np.concatenate([sel, sel | np.uint16(0x8000)])
        pad = (-len(vals)) % 15
        vals = np.concatenate([vals, np.zeros(pad, dtype=np.uint16)]).reshape(-1, 15)
        blk = np.concatenate([np.repeat(top_bits[None, :], vals.shape[0], axis=0), vals], axis=1)
        blocks.append(blk)
    blocks = np.concatenate(blocks)
    blocks = np.concatenate([blocks, np.zeros(((-len(blocks)) % 16, 16), dtype=np.uint16)])
    rows = blocks.reshape(-1, 128)                       # 8 blocks per row, Hkv = 1
    T = rows.shape[0]
    k = torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16)
    v = torch.from_numpy((rows ^ np.uint16(0x8000)).view(np.int16)).view(torch.bfloat16)
    P = 64
    num_pages = (T + P - 1) // P
    slots = torch.arange(T, dtype=torch.int64)
    gpu, ref = _append_both(m, k, v, slots, num_pages, P, 1)
    assert T > 10000
    assert np.array_equal(gpu, ref)


@pytest.mark.parametrize("P", [16, 32, 64, 128])
def test_append_workload_bit_exact_every_page_size(m, P):
    w = workloads.AppendWorkload("append small", 1002 + P, 3000, 3, P, (2 * 3000) // P + 3,
                                 workloads.ValueRecipe(outlier_p=0.01, zero_block_p=0.01))
    k, v = w.kv("cpu")
    slots = w.slot_mapping()
    slots[7] = -1   # skipped token
    gpu, ref = _append_both(m, k, v, slots, w.num_pages, P, 3)
    assert np.array_equal(gpu, ref)


def test_append_with_token_stride_and_fp8(m):
    T, Hkv, P = 500, 2, 16
    g = torch.Generator().manual_seed(5)
    big = (torch.randn(T, 3 * Hkv * 128, generator=g) * 7).to(torch.bfloat16)
    k, v = big[:, :Hkv * 128], big[:, Hkv * 128:2 * Hkv * 128]
    slots = torch.randperm(64 * P, generator=g)[:T].to(torch.int64)
    for dtype in (0, 1):
        cache = m.PagedCache(64, P, Hkv, dtype=dtype)
        kc, vc = big.cuda()[:, :Hkv * 128], big.cuda()[:, Hkv * 128:2 * Hkv * 128]
        m.quantize_append(cache, kc, vc, slots.cuda())
        pool = oracle.OraclePool(64, P, Hkv, dtype=dtype)
        oracle.quantize_append(pool, bits(k.contiguous()), bits(v.contiguous()), slots.numpy())
        torch.cuda.synchronize()
        assert np.array_equal(cache.pool.cpu().numpy(), pool.data), "dtype %d" % dtype


@pytest.mark.parametrize("gk,gv", [(0.5, 2.0), (0.37, 1.9)])
def test_append_with_tensor_scale(m, gk, gv):
    w = workloads.AppendWorkload("append g", 77, 1000, 2, 64, 40, workloads.ValueRecipe(outlier_p=0.02))
    k, v = w.kv("cpu")
    for dtype in (0, 1):
        gpu, ref = _append_both(m, k, v, w.slot_mapping(), w.num_pages, 64, 2, dtype=dtype, gk=gk, gv=gv)
        assert np.array_equal(gpu, ref)


def test_out_of_range_slot_is_skipped_and_reported(m):
    cache = m.PagedCache(2, 16, 1)
    k = torch.ones(3, 1, 128, dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([0, 32, 5], dtype=torch.int64, device="cuda")   # 32 = num_pages * P
    m.quantize_append(cache, k, k, slots)
    assert m.check_device_errors() == -4
    assert m.check_device_errors() == 0          # the word is cleared after a read
    pool = cache.pool.cpu().numpy()
    assert pool[0, 0, 0] != 0 and pool[0, 0, 5 * 64] != 0   # rows 0 and 5 written
