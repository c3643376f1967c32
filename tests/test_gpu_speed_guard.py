"""A coarse speed guard on the decode kernel (32K workload, 2.42 GB of NVFP4 KV).

The kernel runs at its 128-register cap, and an edit anywhere in it can make
ptxas place spill reloads inside the main loop: such builds passed every
numerical test while taking about 1.5x the time (586-614 against 379 us).
This fails when the mean decode-kernel time of 32 launches exceeds 450 us,
which no healthy build on a GB300 comes near (377-382 us measured) and every
such build exceeds."""

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

LIMIT_US = 450.0


def test_decode_kernel_time_on_the_32k_workload():
    import nvfp4_quantised_paged_gb300 as m
    w = workloads.decode_32k()
    cache = m.PagedCache(w.num_pages, w.page_size, w.num_kv_heads)
    for b in range(w.batch):
        k, v = w.seq_kv(b, "cuda")
        m.quantize_append(cache, k, v, w.slots(b).cuda())
    q = w.q("cuda")
    bt, sl = w.block_table.cuda(), w.seq_lens.cuda()
    ws = m.alloc_decode_workspace(cache, w.batch, w.num_q_heads)
    out = torch.empty_like(q)
    for _ in range(4):
        m.paged_decode_attention(cache, q, bt, sl, w.sm_scale, out=out, workspace=ws)
    n = 32
    before = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    after = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    m.profile_decode(before, after)
    torch.cuda.synchronize()
    for _ in range(n):
        m.paged_decode_attention(cache, q, bt, sl, w.sm_scale, out=out, workspace=ws)
    torch.cuda.synchronize()
    m.profile_decode([], [])
    assert m.check_device_errors() == 0
    us = sum(b.elapsed_time(a) for b, a in zip(before, after)) / n * 1e3
    assert us < LIMIT_US, "decode kernel %.1f us per launch on the 32K workload" % us
