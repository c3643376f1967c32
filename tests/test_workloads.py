"""The seeded input generators (workloads/) on the CPU: the same seed gives the
same bits, a sequence regenerates alone, page tables are valid (every page of
the pool used at most once except the shared prefix, rows padded with -1),
the shared prefix is one set of pages and one K/V for every sequence, and the
value recipes have the stated statistics."""

import numpy as np
import pytest
import torch

import workloads


def test_same_seed_same_bits_and_sequences_regenerate_alone():
    w = workloads.make_decode("w", 7, [100, 37, 0, 64], 8, 2, 16)
    k1, v1 = w.seq_kv(1, "cpu")
    k1b, v1b = w.seq_kv(1, "cpu")
    assert torch.equal(k1, k1b) and torch.equal(v1, v1b)
    assert k1.shape == (37, 2, 128) and k1.dtype == torch.bfloat16
    k0, _ = w.seq_kv(0, "cpu")
    assert not torch.equal(k0[:37], k1)           # sequences draw from their own streams
    assert not torch.equal(k1, v1)                # K and V too
    assert torch.equal(w.q("cpu"), workloads.make_decode("w", 7, [100, 37, 0, 64], 8, 2, 16).q("cpu"))
    assert w.seq_kv(2, "cpu")[0].shape[0] == 0


@pytest.mark.parametrize("lens,P,shared", [([100, 37, 0, 64, 1], 16, 0), ([3300, 5000, 3201], 64, 3200)])
def test_page_tables_are_valid(lens, P, shared):
    w = workloads.make_decode("t", 3, lens, 8, 2, P, shared_prefix_tokens=shared, extra_pages=5)
    bt = w.block_table.numpy()
    assert bt.shape[0] == len(lens)
    n_shared = shared // P
    private = []
    for b, n in enumerate(lens):
        need = -(-n // P)
        row = bt[b]
        assert np.all(row[:need] >= 0) and np.all(row[:need] < w.num_pages)
        assert np.all(row[need:] == -1)
        if n_shared:
            assert np.array_equal(row[:n_shared], bt[0, :n_shared])
        private += list(row[n_shared:need])
    assert len(private) == len(set(private))       # private pages used once
    assert not set(private) & set(bt[0, :n_shared])
    slots = w.slots(1)
    assert torch.equal(slots // P, w.block_table[1].to(torch.int64)[torch.arange(lens[1]) // P])
    assert torch.equal(slots % P, torch.arange(lens[1]) % P)


def test_shared_prefix_kv_is_common():
    w = workloads.make_decode("s", 4, [3300, 3264], 8, 2, 64, shared_prefix_tokens=3200)
    k0, v0 = w.seq_kv(0, "cpu")
    k1, v1 = w.seq_kv(1, "cpu")
    assert torch.equal(k0[:3200], k1[:3200]) and torch.equal(v0[:3200], v1[:3200])
    assert not torch.equal(k0[3200:3264], k1[3200:3264])


def test_value_recipes():
    n = 4096
    plain = workloads.draw_kv(n, 2, 9, 0, "cpu", workloads.ValueRecipe(), 0).float()
    assert abs(plain.mean().item()) < 0.02 and abs(plain.std().item() - 1.0) < 0.02
    out = workloads.draw_kv(n, 2, 9, 0, "cpu", workloads.ValueRecipe(outlier_p=0.01), 0).float()
    frac = (out.abs() > 6.0).float().mean().item()   # N(0,1) beyond 6 is ~2e-9; x20 outliers mostly are
    assert 0.006 < frac < 0.011
    zb = workloads.draw_kv(n, 2, 9, 0, "cpu", workloads.ValueRecipe(zero_block_p=0.05), 0)
    blocks = zb.view(n, 2, 8, 16)
    zero = (blocks == 0).all(dim=-1).float().mean().item()
    assert 0.04 < zero < 0.06
    z = blocks[(blocks == 0).all(dim=-1)]
    assert not torch.signbit(z.float()).any()      # zero blocks are +0.0


def test_agent_lengths_and_mix_shapes():
    L = workloads.agent_lengths(1000, 1005, 11)
    assert min(L) >= 3201 and max(L) <= 163_840
    assert 12_000 < float(np.median(L)) < 22_000    # lognormal around 16K
    mix = workloads.agent_mix()
    w = mix.decode
    assert w.batch == 136 and w.shared_prefix_tokens == 3200 and w.page_size == 64
    assert (w.num_q_heads, w.num_kv_heads) == (32, 8)
    for r, p in enumerate(mix.extend_prefix_lens):
        row = mix.num_decode + r
        assert int(w.seq_lens[row]) == p
        s = mix.chunk_slots(r)
        assert s.numel() == mix.chunk_tokens and bool((s >= 0).all())
