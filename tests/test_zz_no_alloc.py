"""The allocation-free decode entry point, for callers that cannot allocate
device memory (a host framework that owns every allocation, or a path where
cudaMalloc's possible device synchronisation is not acceptable).

Through the raw C ABI, two calls in a row must give exactly the bits of the
workspace entry point -- the same kernels on the same inputs -- after a call
of another shape has left its partials in the shared scratch array, and both
must match the fp64 oracle.  The workspace entry point itself is run on a
workspace filled with 0xFF bytes (NaN partials), so a kernel that read scratch
bytes it never wrote would show.  A request larger than the static array is
refused without launching anything.  This file is collected last so that a run
stopping at the first failure has already run every other test."""

import ctypes

import numpy as np
import pytest
import torch

import workloads
from gpu_common import bits, check_attention, decode_both, fill_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import nvfp4_quantised_paged_gb300 as mod
    return mod


def _raw_noalloc(m, cache, q, bt, sl, sm_scale, out, num_splits=0):
    lib = m.library()
    return lib.nvfp4_paged_decode_attention_noalloc(
        cache.desc, ctypes.c_void_p(q.data_ptr()), q.shape[0], q.shape[1], ctypes.c_void_p(bt.data_ptr()),
        bt.shape[1], ctypes.c_void_p(sl.data_ptr()), sm_scale, ctypes.c_void_p(out.data_ptr()), num_splits,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("splits", [0, 5])
def test_noalloc_matches_workspace_entry_point_twice(m, splits):
    # another shape first: its plan and partials stay in the shared array
    w0 = workloads.make_decode("noalloc other shape", 76, [5000, 64, 2000], 16, 2, 64)
    c0, _ = fill_both(w0, m)
    q0 = w0.q("cuda")
    out0 = torch.empty_like(q0)
    assert _raw_noalloc(m, c0, q0, w0.block_table.cuda(), w0.seq_lens.cuda(), w0.sm_scale, out0, 7) == 0

    w = workloads.make_decode("noalloc", 77, [3000, 1, 700, 0, 129], 40, 8, 64,
                              recipe=workloads.ValueRecipe(outlier_p=0.01))
    cache, pool = fill_both(w, m)
    q = w.q("cuda")
    bt, sl = w.block_table.cuda(), w.seq_lens.cuda()
    ws = m.alloc_decode_workspace(cache, w.batch, w.num_q_heads, splits)
    ws.fill_(0xFF)
    ref_gpu = m.paged_decode_attention(cache, q, bt, sl, w.sm_scale, num_splits=splits, workspace=ws)
    _, ref, spread = decode_both(w, m, cache, pool, num_splits=splits)
    check_attention(ref_gpu, ref, "workspace entry point on a 0xFF-filled workspace vs oracle", spread=spread)
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        assert _raw_noalloc(m, cache, q, bt, sl, w.sm_scale, out, splits) == 0
        torch.cuda.synchronize()
        assert m.check_device_errors() == 0
        assert np.array_equal(bits(out), bits(ref_gpu)), "call %d differs from the workspace entry point" % call
        check_attention(out, ref, "noalloc call %d vs oracle" % call, spread=spread)


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
