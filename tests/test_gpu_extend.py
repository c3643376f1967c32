"""Extend attention (section A2, path 2) on the GPU against the fp64 oracle:
ragged prefixes and chunks across the 128-key tile and 256-row CTA
boundaries, GQA groups 1-8, query tiles left empty, the prefix read from the
NVFP4 pages inside the kernel (bit-identical to the workspace path), empty
prefixes and chunks, and the whole path -- prefix dequantised from the NVFP4
cache by prefix_dequant, then attended together with the chunk."""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import EPS_BF16_P, bits, check_attention, fill_both

pytestmark = pytest.mark.gpu
SM = 1.0 / math.sqrt(128)


@pytest.fixture(scope="module")
def m():
    import nvfp4_quantised_paged_gb300 as mod
    return mod


def _rand(shape, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)


def _case(m, prefix_lens, chunk_lens, Hq, Hkv, seed, max_q_len=None):
    cu_p = torch.tensor(np.concatenate([[0], np.cumsum(prefix_lens)]), dtype=torch.int32)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(chunk_lens)]), dtype=torch.int32)
    TQ, TP = int(cu_q[-1]), int(cu_p[-1])
    q = _rand((TQ, Hq, 128), seed)
    kp, vp = _rand((TP, Hkv, 128), seed + 1), _rand((TP, Hkv, 128), seed + 2)
    kn, vn = _rand((TQ, Hkv, 128), seed + 3), _rand((TQ, Hkv, 128), seed + 4)
    out = m.extend_attention(q, kp, vp, cu_p.cuda(), kn, vn, cu_q.cuda(), max_q_len or max(chunk_lens), SM)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    ref = oracle.extend_attention(bits(q), bits(kp), bits(vp), cu_p.numpy(), bits(kn), bits(vn), cu_q.numpy(), SM,
                                  spread=True)
    return out, ref


@pytest.mark.parametrize("prefix_lens,chunk_lens,Hq,Hkv", [
    ([0], [1], 1, 1),
    ([1], [17], 4, 4),
    ([63, 64, 65], [16, 64, 100], 32, 8),
    ([300, 0, 129], [7, 70, 33], 40, 8),
    ([1000], [512], 32, 8),
    ([77, 5], [0, 130], 8, 1),
    ([127, 256, 257, 0], [129, 64, 255, 1], 32, 8),
    ([128, 383], [96, 33], 16, 2),
    ([200, 1030], [40, 9], 32, 2),          # G = 16: a 128-row query tile holds 8 chunk tokens
])
def test_extend_matches_oracle(m, prefix_lens, chunk_lens, Hq, Hkv):
    out, (ref, spread) = _case(m, prefix_lens, chunk_lens, Hq, Hkv, sum(prefix_lens) + sum(chunk_lens) + Hq)
    check_attention(out, ref, "extend %s %s G=%d" % (prefix_lens, chunk_lens, Hq // Hkv), eps=EPS_BF16_P,
                    spread=spread)


def test_chunk_longer_than_bound_is_flagged(m):
    cu = torch.tensor([0, 40], dtype=torch.int32, device="cuda")
    cp = torch.tensor([0, 0], dtype=torch.int32, device="cuda")
    q, kn, vn = _rand((40, 4, 128), 1), _rand((40, 4, 128), 2), _rand((40, 4, 128), 3)
    kp = torch.zeros((1, 4, 128), dtype=torch.bfloat16, device="cuda")
    m.extend_attention(q, kp[:0], kp[:0], cp, kn, vn, cu, 16, SM)
    torch.cuda.synchronize()
    assert m.check_device_errors() == -4


def test_path2_prefix_dequant_then_extend(m):
    """Cached prefixes (NVFP4 pages, shared first pages) -> BF16 workspace ->
    attention of each request's chunk over [workspace rows || chunk]."""
    w = workloads.make_decode("path2", 31, [700, 64, 1500, 100], 32, 8, 64,
                              recipe=workloads.ValueRecipe(outlier_p=0.002), shared_prefix_tokens=64)
    cache, pool = fill_both(w, m)
    lens = w.seq_lens
    cu_p = torch.zeros(w.batch + 1, dtype=torch.int32)
    cu_p[1:] = torch.cumsum(lens, 0)
    kw, vw = m.prefix_dequant(cache, w.block_table.cuda(), lens.cuda(), cu_p.cuda(), int(cu_p[-1]))
    chunk = [50, 512, 1, 130]
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(chunk)]), dtype=torch.int32)
    q = _rand((int(cu_q[-1]), 32, 128), 7)
    kn, vn = _rand((int(cu_q[-1]), 8, 128), 8), _rand((int(cu_q[-1]), 8, 128), 9)
    out = m.extend_attention(q, kw, vw, cu_p.cuda(), kn, vn, cu_q.cuda(), 512, SM)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    rk, rv = oracle.prefix_dequant(pool, w.block_table.numpy(), lens.numpy(), cu_p.numpy())
    assert np.array_equal(bits(kw), rk) and np.array_equal(bits(vw), rv)
    ref, spread = oracle.extend_attention(bits(q), rk, rv, cu_p.numpy(), bits(kn), bits(vn), cu_q.numpy(), SM,
                                          spread=True)
    check_attention(out, ref, "path 2", eps=EPS_BF16_P, spread=spread)


def _paged_case(m, lens, chunk, Hq, Hkv, P, seed, gk=1.0, gv=1.0):
    w = workloads.make_decode("paged extend", seed, lens, Hq, Hkv, P, recipe=workloads.ValueRecipe(outlier_p=0.002))
    cache, pool = fill_both(w, m, gk=gk, gv=gv)
    pl = w.seq_lens
    cu_p = torch.zeros(w.batch + 1, dtype=torch.int32)
    cu_p[1:] = torch.cumsum(pl, 0)
    cu_q = torch.tensor(np.concatenate([[0], np.cumsum(chunk)]), dtype=torch.int32)
    TQ = int(cu_q[-1])
    q = _rand((TQ, Hq, 128), seed + 1)
    kn, vn = _rand((TQ, Hkv, 128), seed + 2), _rand((TQ, Hkv, 128), seed + 3)
    L = max(chunk)
    bt = w.block_table.cuda()
    paged = m.extend_attention_paged(cache, q, bt, pl.cuda(), kn, vn, cu_q.cuda(), L, SM)
    kw, vw = m.prefix_dequant(cache, bt, pl.cuda(), cu_p.cuda(), int(cu_p[-1]))
    two = m.extend_attention(q, kw, vw, cu_p.cuda(), kn, vn, cu_q.cuda(), L, SM)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    return paged, two, (w, pool, pl, cu_p, cu_q, q, kn, vn)


@pytest.mark.parametrize("lens,chunk,Hq,Hkv,P", [
    ([700, 64, 1500, 100], [50, 512, 1, 130], 32, 8, 64),
    ([0, 1, 127, 129, 300], [17, 64, 255, 5, 1], 16, 2, 16),
    ([1000, 257], [96, 200], 40, 8, 128),
    ([63, 2048], [300, 7], 8, 1, 32),
    ([513, 90], [33, 260], 32, 2, 64),
])
def test_paged_extend_equals_dequant_then_extend(m, lens, chunk, Hq, Hkv, P):
    """The prefix expanded inside the kernel gives the same BF16 operands, in the
    same order, as the workspace path: the outputs are identical."""
    paged, two, _ = _paged_case(m, lens, chunk, Hq, Hkv, P, 70 + P)
    assert torch.equal(paged, two)


def test_paged_extend_with_tensor_scales_matches_oracle(m):
    paged, two, (w, pool, pl, cu_p, cu_q, q, kn, vn) = _paged_case(m, [300, 130], [64, 129], 32, 8, 64, 91,
                                                                  gk=0.37, gv=2.5)
    assert torch.equal(paged, two)
    rk, rv = oracle.prefix_dequant(pool, w.block_table.numpy(), pl.numpy(), cu_p.numpy())
    ref, spread = oracle.extend_attention(bits(q), rk, rv, cu_p.numpy(), bits(kn), bits(vn), cu_q.numpy(), SM,
                                          spread=True)
    check_attention(paged, ref, "paged extend g != 1", eps=EPS_BF16_P, spread=spread)


def test_paged_extend_bad_page_is_flagged(m):
    w = workloads.make_decode("paged bad page", 93, [200], 8, 2, 64)
    cache, _ = fill_both(w, m)
    bt = w.block_table.clone()
    bt[0, 1] = -1
    cu_q = torch.tensor([0, 16], dtype=torch.int32, device="cuda")
    q, kn, vn = _rand((16, 8, 128), 94), _rand((16, 2, 128), 95), _rand((16, 2, 128), 96)
    out = m.extend_attention_paged(cache, q, bt.cuda(), w.seq_lens.cuda(), kn, vn, cu_q, 16, SM)
    torch.cuda.synchronize()
    assert m.check_device_errors() == -4
    assert torch.isfinite(out.float()).all()  # the missing page reads as zeros


def test_paged_extend_needs_an_nvfp4_pool(m):
    cache = m.PagedCache(4, 64, 2, dtype=m.DTYPE_FP8_E4M3)
    cu_q = torch.tensor([0, 16], dtype=torch.int32, device="cuda")
    q, kn, vn = _rand((16, 8, 128), 97), _rand((16, 2, 128), 98), _rand((16, 2, 128), 99)
    with pytest.raises(m.NVFP4KVError):
        m.extend_attention_paged(cache, q, torch.zeros((1, 4), dtype=torch.int32, device="cuda"),
                                 torch.tensor([64], dtype=torch.int32, device="cuda"), kn, vn, cu_q, 16, SM)
