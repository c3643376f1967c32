"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (auto split count), on sampled outputs the oracle computes one
(sequence, kv_head) unit at a time from the same BF16 K/V.

  * 32K iso-concurrency decode (batch 64 x 32,768, 64 q / 8 kv heads), with the
    bench step's new token appended at position 32,767 first;
  * 1M long-context decode (batch 2 x 1,048,576, 40 q / 8 kv, channel factors);
  * agent mix (128 sequences of 3.2K-160K tokens sharing a 3,200-token prefix)
    plus its 8 extend requests: prefix dequant of sampled requests bit-exact,
    the 512-token chunk appends bit-exact.
"""

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


def fill(m, w, device="cuda"):
    cache = m.PagedCache(w.num_pages, w.page_size, w.num_kv_heads, device=device)
    if w.shared_prefix_tokens:
        pk, pv = w.prefix_kv(device)
        m.quantize_append(cache, pk, pv, w.slots(0, 0, w.shared_prefix_tokens).to(device))
    for b in range(w.batch):
        k, v = w.private_kv(b, device)
        if k.shape[0]:
            m.quantize_append(cache, k, v, w.slots(b, w.shared_prefix_tokens).to(device))
    return cache


def oracle_unit(w, q, b, kv, k=None, v=None):
    """fp64 attention of the G query heads of (b, kv) over sequence b."""
    if k is None:
        k, v = w.seq_kv(b, "cuda")
    G = w.group
    return oracle.sequence_attention(bits(q[b, kv * G:(kv + 1) * G]), bits(k[:, kv].contiguous()),
                                     bits(v[:, kv].contiguous()), w.sm_scale)


def test_decode_32k_full_size_with_step_append(m):
    w = workloads.decode_32k()
    cache = fill(m, w)
    B, S, Hkv = w.batch, int(w.seq_lens[0]), w.num_kv_heads
    g = torch.Generator(device="cuda")
    g.manual_seed(4242)
    new_k = torch.randn((B, Hkv, 128), generator=g, device="cuda").to(torch.bfloat16)
    new_v = torch.randn((B, Hkv, 128), generator=g, device="cuda").to(torch.bfloat16)
    new_slots = torch.cat([w.slots(b, S - 1, S) for b in range(B)]).cuda()
    m.quantize_append(cache, new_k, new_v, new_slots)
    q = w.q("cuda")
    out = m.paged_decode_attention(cache, q, w.block_table.cuda(), w.seq_lens.cuda(), w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    for b, kv in [(0, 0), (31, 7), (63, 3)]:
        k, v = w.seq_kv(b, "cuda")
        k[S - 1], v[S - 1] = new_k[b], new_v[b]
        ref = oracle_unit(w, q, b, kv, k, v)
        check_attention(out[b, kv * w.group:(kv + 1) * w.group], ref, "32K b=%d kv=%d" % (b, kv))


def test_decode_1m_full_size(m):
    w = workloads.decode_1m()
    cache = fill(m, w)
    q = w.q("cuda")
    out = m.paged_decode_attention(cache, q, w.block_table.cuda(), w.seq_lens.cuda(), w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    del cache
    torch.cuda.empty_cache()
    ref = oracle_unit(w, q, 1, 5)
    check_attention(out[1, 5 * w.group:6 * w.group], ref, "1M b=1 kv=5")


def test_agent_mix_full_size(m):
    mix = workloads.agent_mix()
    w = mix.decode
    cache = fill(m, w)
    q = w.q("cuda")
    dec = list(range(mix.num_decode))
    bt = w.block_table[dec].contiguous()
    out = m.paged_decode_attention(cache, q[dec].contiguous(), bt.cuda(), w.seq_lens[dec].contiguous().cuda(),
                                   w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    lens = w.seq_lens[dec]
    shared = w.shared_prefix_tokens
    casc = m.cascade_decode_attention(cache, q[dec].contiguous(), bt[0, :shared // w.page_size].contiguous().cuda(),
                                      shared, bt.cuda(), lens.contiguous().cuda(), w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    shortest, longest = int(torch.argmin(lens)), int(torch.argmax(lens))
    for b, kv in [(shortest, 1), (longest, 6), (77, 0)]:
        ref = oracle_unit(w, q, b, kv)
        check_attention(out[b, kv * w.group:(kv + 1) * w.group], ref, "agent b=%d kv=%d" % (b, kv))
        check_attention(casc[b, kv * w.group:(kv + 1) * w.group], ref, "agent cascade b=%d kv=%d" % (b, kv))

    # extend requests: dequantise every cached prefix, then append the chunks
    rows = mix.extend_rows()
    pl = w.seq_lens[rows].contiguous()
    cu = torch.zeros(len(rows) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(pl, 0)
    ebt = w.block_table[rows].contiguous()
    kw, vw = m.prefix_dequant(cache, ebt.cuda(), pl.cuda(), cu.cuda(), int(cu[-1]))
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    for r in (0, len(rows) - 1):  # oracle pool of this request's own pages
        row = rows[r]
        k, v = w.seq_kv(row, "cuda")
        n = int(pl[r])
        pool = oracle.OraclePool(-(-n // w.page_size), w.page_size, w.num_kv_heads)
        oracle.quantize_append(pool, bits(k), bits(v), np.arange(n, dtype=np.int64))
        rk, rv = oracle.prefix_dequant(pool, np.arange(pool.num_pages, dtype=np.int32)[None],
                                       np.array([n], dtype=np.int32), np.array([0, n], dtype=np.int32))
        assert np.array_equal(bits(kw[int(cu[r]):int(cu[r + 1])]), rk)
        assert np.array_equal(bits(vw[int(cu[r]):int(cu[r + 1])]), rv)
    # extend attention of every request's 512-token chunk over [its prefix || chunk],
    # sampled tokens against the oracle (a one-token chunk whose "prefix" is the
    # workspace rows followed by the chunk rows before it: the same keys)
    qs = [mix.chunk_q(r, "cuda") for r in range(len(rows))]
    kvs = [mix.chunk_kv(r, "cuda") for r in range(len(rows))]
    L = mix.chunk_tokens
    cu_q = torch.arange(0, L * (len(rows) + 1), L, dtype=torch.int32)
    out = m.extend_attention(torch.cat(qs), kw, vw, cu.cuda(), torch.cat([k for k, _ in kvs]),
                             torch.cat([v for _, v in kvs]), cu_q.cuda(), L, w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    for r, i in ((0, 0), (4, 511), (6, 300)):   # request 4 has the longest prefix
        a, b = int(cu[r]), int(cu[r + 1])
        kpre = torch.cat([kw[a:b], kvs[r][0][:i]])
        vpre = torch.cat([vw[a:b], kvs[r][1][:i]])
        n = kpre.shape[0]
        ref = oracle.extend_attention(bits(qs[r][i:i + 1]), bits(kpre), bits(vpre), np.array([0, n], np.int32),
                                      bits(kvs[r][0][i:i + 1]), bits(kvs[r][1][i:i + 1]), np.array([0, 1], np.int32),
                                      w.sm_scale)
        check_attention(out[r * L + i:r * L + i + 1], ref, "agent extend r=%d token=%d" % (r, i))

    for r in range(len(rows)):
        k, v = mix.chunk_kv(r, "cuda")
        slots = mix.chunk_slots(r)
        m.quantize_append(cache, k, v, slots.cuda())
        if r == 0:  # the chunk's pages against the oracle quantising the same rows
            P = w.page_size
            pages = sorted({int(s) // P for s in slots.tolist()})
            remap = {p: i for i, p in enumerate(pages)}
            pool = oracle.OraclePool(len(pages), P, w.num_kv_heads)
            local = np.array([remap[int(s) // P] * P + int(s) % P for s in slots.tolist()], dtype=np.int64)
            oracle.quantize_append(pool, bits(k), bits(v), local)
            torch.cuda.synchronize()
            got = cache.pool[torch.tensor(pages)].cpu().numpy()
            # compare only the rows the chunk wrote (the first page may hold prefix rows too)
            for t, sl in enumerate(slots.tolist()):
                p, row = remap[sl // P], sl % P
                grp, rr = divmod(row, 16)
                base = grp * 2304
                for h in range(w.num_kv_heads):
                    for off, ln in ((rr * 64, 64), (1024 + rr * 8, 8), (1152 + rr * 64, 64)):
                        assert np.array_equal(got[p, h, base + off:base + off + ln],
                                              pool.data[p, h, base + off:base + off + ln])
                    assert np.array_equal(got[p, h, base + 2176 + rr:base + 2304:16],
                                          pool.data[p, h, base + 2176 + rr:base + 2304:16])
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
