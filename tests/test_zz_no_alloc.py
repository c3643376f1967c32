"""The allocation-free decode entry point, for callers that cannot allocate
device memory (a host framework that owns every allocation, or a path where
cudaMalloc's possible device synchronisation is not acceptable).

It must match the workspace entry point within the attention tolerance of
the other tests, on two calls in a row through the raw C ABI, and reject a
request larger than its static scratch array without launching anything.
This file is collected last so that a run stopping at the first failure has
already run every other test."""

import ctypes

import pytest
import torch

import workloads
from gpu_common import check_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import nvfp4_quantised_paged_gb300 as mod
    return mod


def _fill(m, w):
    cache = m.PagedCache(w.num_pages, w.page_size, w.num_kv_heads)
    for b in range(w.batch):
        k, v = w.seq_kv(b, "cuda")
        if k.shape[0]:
            m.quantize_append(cache, k, v, w.slots(b).cuda())
    return cache


def _raw_noalloc(m, cache, q, bt, sl, sm_scale, out, num_splits=0):
    lib = m.library()
    return lib.nvfp4_paged_decode_attention_noalloc(
        cache.desc, ctypes.c_void_p(q.data_ptr()), q.shape[0], q.shape[1], ctypes.c_void_p(bt.data_ptr()),
        bt.shape[1], ctypes.c_void_p(sl.data_ptr()), sm_scale, ctypes.c_void_p(out.data_ptr()), num_splits,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("splits", [0, 5])
def test_noalloc_matches_workspace_entry_point_twice(m, splits):
    w = workloads.make_decode("noalloc", 77, [3000, 1, 700, 0, 129], 40, 8, 64,
                              recipe=workloads.ValueRecipe(outlier_p=0.01))
    cache = _fill(m, w)
    q = w.q("cuda")
    bt, sl = w.block_table.cuda(), w.seq_lens.cuda()
    ref = m.paged_decode_attention(cache, q, bt, sl, w.sm_scale, num_splits=splits)
    ref_np = ref.float().cpu().double().numpy()
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        assert _raw_noalloc(m, cache, q, bt, sl, w.sm_scale, out, splits) == 0
        torch.cuda.synchronize()
        assert m.check_device_errors() == 0
        check_attention(out, ref_np, "noalloc vs workspace entry point")


def test_noalloc_rejects_requests_beyond_its_scratch(m):
    w = workloads.make_decode("big", 78, [64] * 4096, 64, 8, 64)   # 32,768 (seq, kv_head) pairs
    cache = m.PagedCache(w.num_pages, w.page_size, w.num_kv_heads)
    assert m.decode_workspace_bytes(cache, w.batch, w.num_q_heads) > m.NOALLOC_SCRATCH_BYTES
    q = w.q("cuda")
    out = torch.zeros_like(q)
    rc = _raw_noalloc(m, cache, q, w.block_table.cuda(), w.seq_lens.cuda(), w.sm_scale, out)
    assert rc == -2
    torch.cuda.synchronize()
    assert not out.float().abs().sum().item()   # nothing was launched
