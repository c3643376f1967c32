"""The decode calls captured in a CUDA graph and replayed: the programmatic
launch chains (plan -> decode -> reduce, plan -> shared prefix -> decode ->
reduce) must capture, and every replay must give the eager result, also after
the static inputs are overwritten between replays."""

import pytest
import torch

import workloads
from gpu_common import fill_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import nvfp4_quantised_paged_gb300 as mod
    return mod


def _capture(fn):
    fn()  # first call outside the capture: one-time kernel attributes
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_fused_step_replays_equal_eager(m):
    w = workloads.make_decode("graph fused", 61, [3000, 1, 700, 129, 4097], 32, 8, 64)
    cache = m.PagedCache(w.num_pages, w.page_size, w.num_kv_heads)
    new_k = torch.zeros((w.batch, w.num_kv_heads, 128), dtype=torch.bfloat16, device="cuda")
    new_v = torch.zeros_like(new_k)
    for b in range(w.batch):
        n = int(w.seq_lens[b])
        k, v = w.seq_kv(b, "cuda")
        if n > 1:
            m.quantize_append(cache, k[:n - 1].contiguous(), v[:n - 1].contiguous(), w.slots(b, 0, n - 1).cuda())
        new_k[b], new_v[b] = k[n - 1], v[n - 1]
    q = w.q("cuda")
    bt, sl = w.block_table.cuda(), w.seq_lens.cuda()
    ws = m.alloc_decode_workspace(cache, w.batch, w.num_q_heads)
    out = torch.empty_like(q)

    def step():
        m.paged_decode_attention_append(cache, new_k, new_v, q, bt, sl, w.sm_scale, out=out, workspace=ws)

    g = _capture(step)
    torch.cuda.synchronize()
    eager = out.clone()
    pool = cache.pool.clone()
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    assert torch.equal(out, eager)
    assert torch.equal(cache.pool, pool)  # the appended token is rewritten with the same bytes

    # new queries in the static buffer: the replay attends with them
    q.copy_(workloads.make_decode("graph fused q2", 62, [3000, 1, 700, 129, 4097], 32, 8, 64).q("cuda"))
    g.replay()
    ref = m.paged_decode_attention(cache, q, bt, sl, w.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_cascade_replays_equal_eager(m):
    shared, P = 3200, 64
    w = workloads.make_decode("graph cascade", 63, [3200, 3300, 4000, 3264, 9000] * 4, 32, 8, P,
                              shared_prefix_tokens=shared)
    cache, _ = fill_both(w, m)
    q = w.q("cuda")
    bt, sl = w.block_table.cuda(), w.seq_lens.cuda()
    sp = w.block_table[0, :shared // P].contiguous().cuda()
    ws = torch.empty(m.cascade_workspace_bytes(cache, w.batch, w.num_q_heads, shared), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(q)

    def step():
        m.cascade_decode_attention(cache, q, sp, shared, bt, sl, w.sm_scale, out=out, workspace=ws)

    step()
    torch.cuda.synchronize()
    eager = out.clone()
    g = _capture(step)
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    assert torch.equal(out, eager)

    # shorter sequences in the static length buffer (each within its pages)
    sl.copy_(torch.tensor([3200, 3201, 3900, 3250, 5000] * 4, dtype=torch.int32))
    g.replay()
    ref = m.cascade_decode_attention(cache, q, sp, shared, bt, sl, w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    assert torch.equal(out, ref)
