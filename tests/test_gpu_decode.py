"""GPU parity of paged decode attention against the fp64 oracle (max-abs 2e-2,
rel-L2 3e-3), over page sizes, GQA group sizes (1, 4, 5, 8, 16), ragged and
empty sequences, split counts, the FP8 comparison cache, tensor scales, and
the tiny-decode workload; plus error reporting for bad block-table entries."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import bits, check_attention, decode_both, fill_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import nvfp4_quantised_paged_gb300 as mod
    return mod


def test_tiny_decode_workload(m):
    w = workloads.tiny_decode()
    cache, pool = fill_both(w, m)
    assert np.array_equal(cache.pool.cpu().numpy(), pool.data)
    for splits in (0, 1, 2, 9):
        out, ref, spread = decode_both(w, m, cache, pool, num_splits=splits)
        check_attention(out, ref, "tiny splits=%d" % splits, spread=spread)


@pytest.mark.parametrize("P", [16, 32, 64, 128])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 4), (40, 8), (64, 8), (32, 2)])
def test_decode_page_sizes_and_groups(m, P, Hq, Hkv):
    lens = [1, 63, 64, 65, 300, 1000, 0, 129]
    w = workloads.make_decode("t", 31 + P + Hq, lens, Hq, Hkv, P, recipe=workloads.ValueRecipe(outlier_p=0.01))
    cache, pool = fill_both(w, m)
    out, ref, spread = decode_both(w, m, cache, pool)
    check_attention(out, ref, "P=%d Hq=%d Hkv=%d" % (P, Hq, Hkv), spread=spread)
    assert not out[6].float().abs().sum().item()   # empty sequence -> zeros


# The workload has 63 + 40 + 1 + 1 = 105 chunks of 64 tokens per kv head, so
# U = 210 units: 104 and 105 splits give every CTA >= 2 units (the reduction
# takes interior CTAs' partials without recomputing their ranges), 106 gives
# some CTAs one unit, 210 exactly one each, 211 and 500 leave CTAs empty.
@pytest.mark.parametrize("splits", [1, 3, 7, 64, 104, 105, 106, 210, 211, 500])
def test_split_count_does_not_change_the_result_beyond_tolerance(m, splits):
    w = workloads.make_decode("s", 5, [4000, 2500, 31, 1], 16, 2, 64)
    cache, pool = fill_both(w, m)
    out, ref, spread = decode_both(w, m, cache, pool, num_splits=splits)
    check_attention(out, ref, "splits=%d" % splits, spread=spread)


# Batches of up to 96 sequences are planned inside every decode CTA (two
# sequences per thread of the 64-thread CTA, the reduction scanning seq_lens in
# each warp), larger ones by the plan kernel: both sides of the threshold, with
# ragged and empty sequences, and the launch count of each.
@pytest.mark.parametrize("B", [1, 33, 95, 96, 97, 160])
def test_batch_planned_in_cta_and_by_plan_kernel(m, B):
    rng = np.random.default_rng(700 + B)
    lens = [int(x) for x in rng.integers(1, 400, size=B)]
    if B > 1:
        lens[B // 2] = 0
    w = workloads.make_decode("plan%d" % B, 700 + B, lens, 16, 2, 32)
    cache, pool = fill_both(w, m)
    assert m.decode_launch_count(cache, B, 16) == (2 if B <= 96 else 3)
    out, ref, spread = decode_both(w, m, cache, pool)
    check_attention(out, ref, "B=%d" % B, spread=spread)
    assert m.check_device_errors() == 0
    # a length beyond the block table is clamped and flagged either way
    sl = w.seq_lens.clone()
    sl[B - 1] = w.block_table.shape[1] * 32 + 5
    m.paged_decode_attention(cache, w.q("cuda"), w.block_table.cuda(), sl.cuda())
    assert m.check_device_errors() == -4


def test_channel_outliers_long_sequence(m):
    w = workloads.make_decode("c", 6, [20000, 7], 40, 8, 64, recipe=workloads.ValueRecipe(channel_lognormal=True))
    cache, pool = fill_both(w, m)
    out, ref, spread = decode_both(w, m, cache, pool)
    check_attention(out, ref, "channel outliers", spread=spread)


def test_shared_prefix_pages(m):
    w = workloads.make_decode("p", 8, [3300, 5000, 3201, 4000], 32, 8, 64, shared_prefix_tokens=3200)
    cache, pool = fill_both(w, m)
    out, ref, spread = decode_both(w, m, cache, pool)
    check_attention(out, ref, "shared prefix", spread=spread)


@pytest.mark.parametrize("P,Hq,Hkv", [(16, 32, 4), (64, 32, 4), (128, 32, 4), (64, 32, 2), (16, 16, 1), (64, 40, 8)])
def test_fp8_cache_decode(m, P, Hq, Hkv):
    """G = 8 and 5 take one 8-wide N tile of the FP8 kernel, G = 16 two."""
    w = workloads.make_decode("f", 9 + P + Hq, [1, 100, 2000, 64], Hq, Hkv, P,
                              recipe=workloads.ValueRecipe(outlier_p=0.01))
    cache, pool = fill_both(w, m, dtype=1)
    assert np.array_equal(cache.pool.cpu().numpy(), pool.data)
    out, ref, spread = decode_both(w, m, cache, pool)
    check_attention(out, ref, "fp8 P=%d G=%d" % (P, Hq // Hkv), spread=spread)


def test_tensor_scales_and_custom_sm_scale(m):
    w = workloads.make_decode("g", 10, [700, 33], 16, 2, 32)
    cache, pool = fill_both(w, m, gk=0.75, gv=3.0)
    q = w.q("cuda")
    out = m.paged_decode_attention(cache, q, w.block_table.cuda(), w.seq_lens.cuda(), sm_scale=0.3)
    ref, spread = oracle.decode_attention(pool, bits(q), w.block_table.numpy(), w.seq_lens.numpy(), 0.3, spread=True)
    check_attention(out, ref, "tensor scales", spread=spread)


def test_large_query_values(m):
    """Q far outside FP16 range is pre-scaled by a power of two per head."""
    w = workloads.make_decode("q", 11, [500], 8, 1, 16)
    cache, pool = fill_both(w, m)
    q = (w.q("cuda").float() * 3.0e5).to(torch.bfloat16)
    q[0, 3] = (q[0, 3].float() * 1e-30).to(torch.bfloat16)
    out = m.paged_decode_attention(cache, q, w.block_table.cuda(), w.seq_lens.cuda(), sm_scale=1e-6)
    ref, spread = oracle.decode_attention(pool, bits(q), w.block_table.numpy(), w.seq_lens.numpy(), 1e-6, spread=True)
    check_attention(out, ref, "large q", spread=spread)


def test_bad_block_table_entry_is_reported_not_read(m):
    w = workloads.make_decode("bad", 12, [200, 300], 8, 2, 16)
    cache, pool = fill_both(w, m)
    bt = w.block_table.clone()
    bt[1, 3] = w.num_pages + 1000     # out of range: the kernel must skip it and flag it
    bt[0, 2] = -7
    out = m.paged_decode_attention(cache, w.q("cuda"), bt.cuda(), w.seq_lens.cuda())
    assert m.check_device_errors() == -4
    assert m.check_device_errors() == 0
    assert torch.isfinite(out.float()).all()


def test_seq_len_beyond_table_is_clamped_and_reported(m):
    w = workloads.make_decode("len", 13, [40], 4, 1, 16)
    cache, pool = fill_both(w, m)
    sl = torch.tensor([10_000], dtype=torch.int32, device="cuda")
    m.paged_decode_attention(cache, w.q("cuda"), w.block_table.cuda(), sl)
    assert m.check_device_errors() == -4
