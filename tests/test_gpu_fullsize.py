"""Parity at the benchmark's full sizes, on FULL outputs: every (sequence, kv
head) unit, every extend row and the whole append pool, computed by the oracle
from the same BF16 bits on all host cores (ctypes releases the GIL, so the
units run in parallel threads).

  * 32K iso-concurrency decode (batch 64 x 32,768, 64 q / 8 kv heads) through
    the exact call bench.py times: paged_decode_attention_append with the
    automatic split, each sequence's new token quantised into position 32,767
    in the same launch (the 64 new rows bit-exact too);
  * 1M long-context decode (batch 2 x 1,048,576, 40 q / 8 kv, channel factors),
    automatic split;
  * the 32K and 1M workloads over the FP8-E4M3 comparison cache, automatic split;
  * agent mix: the 128 decode sequences (3.2K-160K tokens sharing a 3,200-token
    prefix) through plain and cascade decode; the 8 extend requests' prefix
    dequant bit-exact, their extend attention on all 8 x 512 chunk rows over the
    oracle's own workspace, the paged-prefix extend bit-identical to it, and the
    chunks' appends bit-exact;
  * quantise-append of 65,536 tokens x 8 kv heads through a random slot mapping
    into 64-token pages: the whole 151 MB pool bit-exact.
"""

import concurrent.futures
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import EPS_BF16_P, bits, check_attention

pytestmark = pytest.mark.gpu

THREADS = os.cpu_count() or 1


@pytest.fixture(scope="module")
def m():
    import nvfp4_quantised_paged_gb300 as mod
    return mod


@pytest.fixture(scope="module")
def pool_exec():
    with concurrent.futures.ThreadPoolExecutor(max_workers=THREADS) as ex:
        yield ex


def fill(m, w, device="cuda", dtype=None):
    cache = m.PagedCache(w.num_pages, w.page_size, w.num_kv_heads, device=device,
                         dtype=m.DTYPE_NVFP4 if dtype is None else dtype)
    if w.shared_prefix_tokens:
        pk, pv = w.prefix_kv(device)
        m.quantize_append(cache, pk, pv, w.slots(0, 0, w.shared_prefix_tokens).to(device))
    for b in range(w.batch):
        k, v = w.private_kv(b, device)
        if k.shape[0]:
            m.quantize_append(cache, k, v, w.slots(b, w.shared_prefix_tokens).to(device))
    return cache


def rows_mask(local_slots, pool):
    """Boolean mask of the NVFP4 pool bytes that hold the rows at `local_slots`
    (16-token groups of 2,304 bytes: K codes, K scales, V codes, V scales [8][16])."""
    mask = np.zeros(pool.data.shape, dtype=bool)
    for s in np.asarray(local_slots).tolist():
        p, row = divmod(int(s), pool.page_size)
        grp, rr = divmod(row, 16)
        base = grp * 2304
        for off, ln in ((rr * 64, 64), (1024 + rr * 8, 8), (1152 + rr * 64, 64)):
            mask[p, :, base + off:base + off + ln] = True
        mask[p, :, base + 2176 + rr:base + 2304:16] = True
    return mask


def oracle_decode_all(ex, w, q, seqs, new_kv=None, window=3, dtype=oracle.DTYPE_NVFP4):
    """fp64 attention (and spread) of every (sequence, kv head) unit of the
    sequences `seqs`, each computed by the oracle from sequence b's BF16 K/V as
    drawn on the GPU (the product's own inputs).  new_kv = (k_new, v_new)
    replaces each sequence's last token.  Returns (ref, spread) [len(seqs)][Hq][128]."""
    G, Hkv = w.group, w.num_kv_heads
    qb = bits(q)
    ref = np.zeros((len(seqs), w.num_q_heads, 128))
    spread = np.zeros_like(ref)
    pending = []

    def unit(i, kv, kb, vb, qg):
        return i, kv, oracle.sequence_attention(qg, kb, vb, w.sm_scale, dtype=dtype, spread=True)

    def drain(keep):
        while len(pending) > keep:
            for f in pending.pop(0):
                i, kv, (o, s) = f.result()
                ref[i, kv * G:(kv + 1) * G], spread[i, kv * G:(kv + 1) * G] = o, s

    for i, b in enumerate(seqs):
        k, v = w.seq_kv(b, "cuda")
        if new_kv is not None:
            k[-1], v[-1] = new_kv[0][b], new_kv[1][b]
        futs = [ex.submit(unit, i, kv, bits(k[:, kv].contiguous()), bits(v[:, kv].contiguous()),
                          qb[b, kv * G:(kv + 1) * G].copy()) for kv in range(Hkv)]
        del k, v
        pending.append(futs)
        drain(window)     # bounds the host copies in flight
    drain(0)
    return ref, spread


def test_decode_32k_full_output_of_the_bench_call(m, pool_exec):
    w = workloads.decode_32k()
    cache = fill(m, w)
    B, S, Hkv = w.batch, int(w.seq_lens[0]), w.num_kv_heads
    g = torch.Generator(device="cuda")
    g.manual_seed(4242)   # the bench step's new tokens
    new_k = torch.randn((B, Hkv, 128), generator=g, device="cuda").to(torch.bfloat16)
    new_v = torch.randn((B, Hkv, 128), generator=g, device="cuda").to(torch.bfloat16)
    q = w.q("cuda")
    out = m.paged_decode_attention_append(cache, new_k, new_v, q, w.block_table.cuda(), w.seq_lens.cuda(),
                                          w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0

    # the 64 new rows, bit-exact: the oracle quantises the new tokens into a pool of their pages
    slots = torch.cat([w.slots(b, S - 1, S) for b in range(B)])
    pages = (slots // w.page_size).tolist()
    local = np.array([i * w.page_size + int(s) % w.page_size for i, s in enumerate(slots.tolist())], np.int64)
    small = oracle.OraclePool(B, w.page_size, Hkv)
    oracle.quantize_append(small, bits(new_k), bits(new_v), local)
    mask = rows_mask(local, small)
    assert np.array_equal(cache.pool[torch.tensor(pages)].cpu().numpy()[mask], small.data[mask])

    ref, spread = oracle_decode_all(pool_exec, w, q, list(range(B)), new_kv=(new_k, new_v))
    check_attention(out, ref, "32K full output (fused append + decode, auto split)", spread=spread)


def test_decode_32k_fp8_cache_full_output(m, pool_exec):
    """The FP8-E4M3 comparison cache at the 32K workload, through the call the
    bench times for it (paged_decode_attention, automatic split): every unit."""
    w = workloads.decode_32k()
    cache = fill(m, w, dtype=m.DTYPE_FP8_E4M3)
    q = w.q("cuda")
    out = m.paged_decode_attention(cache, q, w.block_table.cuda(), w.seq_lens.cuda(), w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    del cache
    torch.cuda.empty_cache()
    ref, spread = oracle_decode_all(pool_exec, w, q, list(range(w.batch)), dtype=oracle.DTYPE_FP8)
    check_attention(out, ref, "32K FP8 cache full output (auto split)", spread=spread)


def test_decode_1m_full_output(m, pool_exec):
    w = workloads.decode_1m()
    cache = fill(m, w)
    q = w.q("cuda")
    out = m.paged_decode_attention(cache, q, w.block_table.cuda(), w.seq_lens.cuda(), w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    del cache
    torch.cuda.empty_cache()
    ref, spread = oracle_decode_all(pool_exec, w, q, [0, 1], window=1)
    check_attention(out, ref, "1M full output (auto split)", spread=spread)


def test_decode_1m_fp8_cache_full_output(m, pool_exec):
    """The FP8-E4M3 comparison cache at the 1M workload (4.3 GB of FP8 KV): every unit."""
    w = workloads.decode_1m()
    cache = fill(m, w, dtype=m.DTYPE_FP8_E4M3)
    q = w.q("cuda")
    out = m.paged_decode_attention(cache, q, w.block_table.cuda(), w.seq_lens.cuda(), w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    del cache
    torch.cuda.empty_cache()
    ref, spread = oracle_decode_all(pool_exec, w, q, [0, 1], window=1, dtype=oracle.DTYPE_FP8)
    check_attention(out, ref, "1M FP8 cache full output (auto split)", spread=spread)


def test_agent_mix_full_output(m, pool_exec):
    mix = workloads.agent_mix()
    w = mix.decode
    P, Hkv = w.page_size, w.num_kv_heads
    cache = fill(m, w)
    q = w.q("cuda")
    dec = list(range(mix.num_decode))
    bt = w.block_table[dec].contiguous()
    lens = w.seq_lens[dec].contiguous()
    qd = q[dec].contiguous()
    out = m.paged_decode_attention(cache, qd, bt.cuda(), lens.cuda(), w.sm_scale)
    shared = w.shared_prefix_tokens
    casc = m.cascade_decode_attention(cache, qd, bt[0, :shared // P].contiguous().cuda(), shared, bt.cuda(),
                                      lens.cuda(), w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    ref, spread = oracle_decode_all(pool_exec, w, q, dec)
    check_attention(out, ref, "agent mix decode, all 128 sequences", spread=spread)
    check_attention(casc, ref, "agent mix cascade decode, all 128 sequences", spread=spread)

    # path 2 of the 8 extend requests: the prefix workspace against the oracle's own
    rows = mix.extend_rows()
    pl = w.seq_lens[rows].contiguous()
    cu = torch.zeros(len(rows) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(pl, 0)
    kw, vw = m.prefix_dequant(cache, w.block_table[rows].contiguous().cuda(), pl.cuda(), cu.cuda(), int(cu[-1]))
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0

    def oracle_prefix(r):
        k, v = host_kv[r]
        n = int(pl[r])
        pool = oracle.OraclePool(-(-n // P), P, Hkv)
        oracle.quantize_append(pool, k, v, np.arange(n, dtype=np.int64))
        return oracle.prefix_dequant(pool, np.arange(pool.num_pages, dtype=np.int32)[None],
                                     np.array([n], dtype=np.int32), np.array([0, n], dtype=np.int32))

    host_kv = []
    for row in rows:
        k, v = w.seq_kv(row, "cuda")
        host_kv.append((bits(k), bits(v)))
    parts = list(pool_exec.map(oracle_prefix, range(len(rows))))
    del host_kv
    rk = np.concatenate([a for a, _ in parts])
    rv = np.concatenate([b for _, b in parts])
    assert np.array_equal(bits(kw), rk) and np.array_equal(bits(vw), rv), "prefix workspace differs"

    qs = torch.cat([mix.chunk_q(r, "cuda") for r in range(len(rows))])
    kvs = [mix.chunk_kv(r, "cuda") for r in range(len(rows))]
    kn, vn = torch.cat([k for k, _ in kvs]), torch.cat([v for _, v in kvs])
    L = mix.chunk_tokens
    cu_q = torch.arange(0, L * (len(rows) + 1), L, dtype=torch.int32)
    ext = m.extend_attention(qs, kw, vw, cu.cuda(), kn, vn, cu_q.cuda(), L, w.sm_scale)
    # the same extends with the prefix read from the NVFP4 pages inside the kernel: identical
    paged = m.extend_attention_paged(cache, qs, w.block_table[rows].contiguous().cuda(), pl.cuda(), kn, vn,
                                     cu_q.cuda(), L, w.sm_scale)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    assert torch.equal(paged, ext), "paged-prefix extend differs from dequant + extend"
    del paged
    eref, espread = oracle.extend_attention(bits(qs), rk, rv, cu.numpy(), bits(kn), bits(vn), cu_q.numpy(),
                                            w.sm_scale, nthreads=THREADS, spread=True)
    check_attention(ext, eref, "agent mix extend, all 8 x 512 rows", eps=EPS_BF16_P, spread=espread)

    # the chunks' appends: each chunk's rows bit-exact in the pool
    slots = torch.cat([mix.chunk_slots(r) for r in range(len(rows))])
    m.quantize_append(cache, kn, vn, slots.cuda())
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    pages = sorted({int(s) // P for s in slots.tolist()})
    remap = {p: i for i, p in enumerate(pages)}
    pool = oracle.OraclePool(len(pages), P, Hkv)
    local = np.array([remap[int(s) // P] * P + int(s) % P for s in slots.tolist()], dtype=np.int64)
    oracle.quantize_append(pool, bits(kn), bits(vn), local)
    mask = rows_mask(local, pool)    # the first page of a chunk may also hold prefix rows
    assert np.array_equal(cache.pool[torch.tensor(pages)].cpu().numpy()[mask], pool.data[mask]), \
        "chunk appends differ"


def test_append_65k_whole_pool(m, pool_exec):
    w = workloads.append_65k()
    k, v = w.kv("cuda")
    slots = w.slot_mapping()
    cache = m.PagedCache(w.num_pages, w.page_size, w.num_kv_heads)
    m.quantize_append(cache, k, v, slots.cuda())
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    pool = oracle.OraclePool(w.num_pages, w.page_size, w.num_kv_heads)
    kb, vb, sl = bits(k), bits(v), slots.numpy()
    # token ranges in parallel: distinct tokens write distinct slots of the one pool
    step = -(-w.num_tokens // THREADS)
    list(pool_exec.map(lambda s: oracle.quantize_append(pool, kb[s:s + step], vb[s:s + step], sl[s:s + step]),
                       range(0, w.num_tokens, step)))
    got = cache.pool.cpu().numpy()
    assert got.shape == pool.data.shape
    diff = np.argwhere(got != pool.data)
    assert diff.size == 0, "%d bytes differ, first at %s" % (len(diff), diff[:3].tolist())
