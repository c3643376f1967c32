"""Cascade decode (the shared prefix attended once per kv head for all
sequences, merged by log-sum-exp with each sequence's own part) against the
fp64 oracle's plain decode attention and against the GPU's plain decode:
page sizes 16, 32, 64 and 128, groups of 1, 2, 4, 5, 8 and 16 query heads,
suffixes of 0 to thousands of tokens, explicit split counts, tensor scales,
a sequence shorter than the shared prefix (flagged), and the FP8 pool
(unsupported)."""

import pytest
import torch

import oracle
import workloads
from gpu_common import check_attention, decode_both, fill_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import nvfp4_quantised_paged_gb300 as mod
    return mod


@pytest.mark.parametrize("lens,shared,Hq,Hkv,P,splits,gk,gv", [
    ([3200, 3300, 4000, 3264, 9000], 3200, 32, 8, 64, 0, 1.0, 1.0),
    ([128, 129, 1000, 128], 128, 40, 8, 16, 0, 1.0, 1.0),
    ([640] * 70 + [700, 2000], 640, 64, 8, 64, 0, 1.0, 1.0),
    ([256, 300, 511], 256, 8, 2, 16, 5, 1.0, 1.0),
    ([512, 515, 900, 2048], 512, 8, 8, 32, 0, 1.0, 1.0),          # G = 1, P = 32
    ([256, 257, 700] * 3, 256, 32, 2, 128, 0, 1.0, 1.0),          # G = 16 (two N tiles), P = 128
    ([192, 200, 1500, 4000], 192, 4, 2, 64, 3, 0.37, 2.5),        # G = 2, tensor scales
])
def test_cascade_matches_oracle_and_plain_decode(m, lens, shared, Hq, Hkv, P, splits, gk, gv):
    w = workloads.make_decode("cascade", 51 + shared, lens, Hq, Hkv, P, shared_prefix_tokens=shared,
                              recipe=workloads.ValueRecipe(outlier_p=0.003))
    cache, pool = fill_both(w, m, gk=gk, gv=gv)
    plain, ref, spread = decode_both(w, m, cache, pool, num_splits=splits)
    q = w.q("cuda")
    shared_pages = w.block_table[0, :shared // P].contiguous().cuda()
    out = m.cascade_decode_attention(cache, q, shared_pages, shared, w.block_table.cuda(), w.seq_lens.cuda(),
                                     w.sm_scale, num_splits=splits)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    check_attention(out, ref, "cascade vs oracle", spread=spread)
    check_attention(out, plain.float().cpu().double().numpy(), "cascade vs plain decode", spread=spread,
                    both_rounded=True)


def test_sequence_shorter_than_the_shared_prefix_is_flagged(m):
    w = workloads.make_decode("short", 52, [256, 256], 8, 2, 64, shared_prefix_tokens=256)
    cache, _ = fill_both(w, m)
    lens = w.seq_lens.clone()
    lens[1] = 100
    m.cascade_decode_attention(cache, w.q("cuda"), w.block_table[0, :4].contiguous().cuda(), 256,
                               w.block_table.cuda(), lens.cuda(), w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == -4


def test_fp8_pool_is_unsupported(m):
    w = workloads.make_decode("fp8", 53, [128, 192], 8, 2, 64, shared_prefix_tokens=128)
    cache = m.PagedCache(w.num_pages, 64, 2, dtype=m.DTYPE_FP8_E4M3)
    with pytest.raises(m.NVFP4KVError):
        m.cascade_decode_attention(cache, w.q("cuda"), w.block_table[0, :2].contiguous().cuda(), 128,
                                   w.block_table.cuda(), w.seq_lens.cuda(), w.sm_scale)
