"""The fused decode step (new token appended in the decode launch) against the
two-call path it replaces (quantise-append of the token, then decode): the
pools must be bit-identical and the outputs identical, over NVFP4 and FP8
caches, tensor scales, page sizes 16 to 128, groups of 1, 4 and 16 query heads
(both N-tile instances of each cache format), tokens landing on a page's first
row, single-token and empty sequences, many sequence ends per CTA, strided
token rows, explicit split counts, and a bad block-table entry; plus the
fused result against the fp64 oracle."""

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


def _prepare(m, w, dtype, gk, gv, seed):
    """Two identical caches holding every sequence but its last token, and the last tokens."""
    caches = [m.PagedCache(w.num_pages, w.page_size, w.num_kv_heads, dtype=dtype, k_global_scale=gk,
                           v_global_scale=gv) for _ in range(2)]
    new_k = torch.zeros((w.batch, w.num_kv_heads, 128), dtype=torch.bfloat16, device="cuda")
    new_v = torch.zeros_like(new_k)
    for b in range(w.batch):
        n = int(w.seq_lens[b])
        if n == 0:
            continue
        k, v = w.seq_kv(b, "cuda")
        if n > 1:
            for c in caches:
                m.quantize_append(c, k[:n - 1].contiguous(), v[:n - 1].contiguous(), w.slots(b, 0, n - 1).cuda())
        new_k[b], new_v[b] = k[n - 1], v[n - 1]
    return caches, new_k, new_v


def _two_calls(m, w, cache, new_k, new_v, q, num_splits=0):
    lens = w.seq_lens
    live = [b for b in range(w.batch) if int(lens[b]) > 0]
    slots = torch.cat([w.slots(b, int(lens[b]) - 1, int(lens[b])) for b in live]).cuda()
    m.quantize_append(cache, new_k[live].contiguous(), new_v[live].contiguous(), slots)
    return m.paged_decode_attention(cache, q, w.block_table.cuda(), lens.cuda(), w.sm_scale, num_splits=num_splits)


@pytest.mark.parametrize("dtype,gk,gv,P,lens,splits,Hq,Hkv", [
    (0, 1.0, 1.0, 64, [3000, 1, 64, 65, 0, 700, 129], 0, 32, 8),
    (0, 0.7, 2.5, 16, [17, 16, 33, 1000, 2], 0, 32, 8),
    (1, 1.0, 1.0, 64, [513, 64, 1], 0, 32, 8),
    (0, 1.0, 1.0, 32, [5000, 33, 97], 7, 32, 8),
    (0, 1.0, 1.0, 128, [129, 2000, 1, 128], 0, 32, 2),    # G = 16: the two-N-tile instance
    (1, 0.5, 4.0, 64, [700, 65, 3], 0, 32, 2),            # FP8, G = 16, tensor scales
    (0, 1.0, 1.0, 64, [900, 64, 2], 0, 8, 8),             # G = 1
])
def test_fused_equals_append_then_decode(m, dtype, gk, gv, P, lens, splits, Hq, Hkv):
    w = workloads.make_decode("fused", 41 + P, lens, Hq, Hkv, P, recipe=workloads.ValueRecipe(outlier_p=0.003))
    (c_fused, c_two), new_k, new_v = _prepare(m, w, dtype, gk, gv, 41)
    q = w.q("cuda")
    out_f = m.paged_decode_attention_append(c_fused, new_k, new_v, q, w.block_table.cuda(), w.seq_lens.cuda(),
                                            w.sm_scale, num_splits=splits)
    out_t = _two_calls(m, w, c_two, new_k, new_v, q, splits)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    assert torch.equal(c_fused.pool, c_two.pool)
    assert torch.equal(out_f, out_t)


def test_many_sequence_ends_per_cta_and_strided_rows(m):
    rng = np.random.default_rng(9)
    lens = [int(x) for x in rng.integers(1, 200, size=300)]
    w = workloads.make_decode("many ends", 43, lens, 8, 4, 16)
    (c_fused, c_two), new_k, new_v = _prepare(m, w, 0, 1.0, 1.0, 43)
    wide = torch.zeros((w.batch, 3, 4 * 128), dtype=torch.bfloat16, device="cuda")   # fused QKV-like rows
    wide[:, 1] = new_k.reshape(w.batch, -1)
    wide[:, 2] = new_v.reshape(w.batch, -1)
    q = w.q("cuda")
    out_f = m.paged_decode_attention_append(c_fused, wide[:, 1], wide[:, 2], q, w.block_table.cuda(),
                                            w.seq_lens.cuda(), w.sm_scale)
    out_t = _two_calls(m, w, c_two, new_k, new_v, q)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    assert torch.equal(c_fused.pool, c_two.pool)
    assert torch.equal(out_f, out_t)


def test_fused_matches_oracle(m):
    w = workloads.make_decode("fused oracle", 44, [1500, 1, 64, 300], 40, 8, 64)
    (c_fused, _), new_k, new_v = _prepare(m, w, 0, 1.0, 1.0, 44)
    q = w.q("cuda")
    out = m.paged_decode_attention_append(c_fused, new_k, new_v, q, w.block_table.cuda(), w.seq_lens.cuda(),
                                          w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    pool = oracle.OraclePool(w.num_pages, w.page_size, w.num_kv_heads)
    for b in range(w.batch):
        k, v = w.seq_kv(b, "cuda")
        oracle.quantize_append(pool, bits(k), bits(v), w.slots(b).numpy())
    assert np.array_equal(c_fused.pool.cpu().numpy(), pool.data)
    ref, spread = oracle.decode_attention(pool, bits(q), w.block_table.numpy(), w.seq_lens.numpy(), w.sm_scale,
                                          spread=True)
    check_attention(out, ref, "fused decode", spread=spread)


def test_bad_page_for_the_new_token_is_flagged(m):
    w = workloads.make_decode("bad", 45, [100, 70], 8, 2, 64)
    (c_fused, _), new_k, new_v = _prepare(m, w, 0, 1.0, 1.0, 45)
    bt = w.block_table.clone()
    bt[1, 1] = w.num_pages + 5          # the page holding token 69 of sequence 1
    m.paged_decode_attention_append(c_fused, new_k, new_v, w.q("cuda"), bt.cuda(), w.seq_lens.cuda(), w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == -4
