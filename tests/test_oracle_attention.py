"""Pins for the oracle's fp64 decode attention and prefix dequant.

Grid-valued K/V survive quantisation unchanged, so the oracle's paged
attention over them must equal torch's own scaled_dot_product_attention in
float64 (a library routine, with its GQA head mapping) on the raw values.
Closed forms cover one token, identical keys and two tokens; invariants
cover the physical placement of pages.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle_helpers import bf16_bits_to_f64, grid_rows, to_bf16_bits

SM = 1.0 / math.sqrt(128)


def build_cache(rng, seq_lens, Hkv, P, num_pages=None, dtype=oracle.DTYPE_NVFP4, grid=True):
    """Random placement of each sequence's pages; returns pool, block table, K, V (float64)."""
    counts = [-(-n // P) for n in seq_lens]
    num_pages = num_pages or sum(counts) + 3
    perm = rng.permutation(num_pages)
    bt = np.full((len(seq_lens), max(counts + [1])), -1, dtype=np.int32)
    pos = 0
    for b, c in enumerate(counts):
        bt[b, :c] = perm[pos:pos + c]
        pos += c
    pool = oracle.OraclePool(num_pages, P, Hkv, dtype=dtype)
    ks, vs = [], []
    for b, n in enumerate(seq_lens):
        if grid:
            k = grid_rows(rng, n * Hkv).reshape(n, Hkv, 128)
            v = grid_rows(rng, n * Hkv).reshape(n, Hkv, 128)
        else:
            k = bf16_bits_to_f64(to_bf16_bits(rng.standard_normal((n, Hkv, 128))))
            v = bf16_bits_to_f64(to_bf16_bits(rng.standard_normal((n, Hkv, 128))))
        t = np.arange(n)
        slots = (bt[b, t // P].astype(np.int64) * P + t % P)
        oracle.quantize_append(pool, to_bf16_bits(k), to_bf16_bits(v), slots)
        ks.append(k)
        vs.append(v)
    return pool, bt, ks, vs


@pytest.mark.parametrize("Hq,Hkv,P,lens", [
    (4, 1, 16, [256, 300]),
    (8, 2, 16, [1, 17, 40]),
    (40, 8, 64, [70, 129]),
    (64, 8, 32, [33]),
])
def test_paged_attention_equals_torch_sdpa_on_grid_values(Hq, Hkv, P, lens):
    rng = np.random.default_rng(sum(lens) + Hq)
    pool, bt, ks, vs = build_cache(rng, lens, Hkv, P)
    q_bits = to_bf16_bits(rng.standard_normal((len(lens), Hq, 128)))
    out = oracle.decode_attention(pool, q_bits, bt, np.array(lens, dtype=np.int32), SM, nthreads=4)
    qf = torch.from_numpy(bf16_bits_to_f64(q_bits))
    for b, n in enumerate(lens):
        qb = qf[b][None, :, None, :]                                       # [1][Hq][1][D]
        kb = torch.from_numpy(ks[b]).permute(1, 0, 2)[None]                # [1][Hkv][n][D]
        vb = torch.from_numpy(vs[b]).permute(1, 0, 2)[None]
        ref = F.scaled_dot_product_attention(qb, kb, vb, scale=SM, enable_gqa=True)[0, :, 0, :]
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(7)
    pool, bt, ks, vs = build_cache(rng, [1, 1], 2, 16)
    q = to_bf16_bits(rng.standard_normal((2, 6, 128)))
    out = oracle.decode_attention(pool, q, bt, np.array([1, 1], dtype=np.int32), SM)
    for b in range(2):
        for h in range(6):
            assert np.array_equal(out[b, h], vs[b][0, h // 3])


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(8)
    n, P = 50, 16
    pool = oracle.OraclePool(8, P, 1)
    krow = grid_rows(rng, 1)
    k = np.repeat(krow, n, axis=0)
    v = grid_rows(rng, n)
    oracle.quantize_append(pool, to_bf16_bits(k), to_bf16_bits(v), np.arange(n, dtype=np.int64))
    bt = np.arange(4, dtype=np.int32)[None]
    out = oracle.decode_attention(pool, to_bf16_bits(rng.standard_normal((1, 3, 128))), bt,
                                  np.array([n], dtype=np.int32), SM)
    for h in range(3):
        np.testing.assert_allclose(out[0, h], v.mean(axis=0), rtol=1e-13, atol=1e-13)


def test_two_tokens_blend_by_logistic_weight():
    rng = np.random.default_rng(9)
    pool = oracle.OraclePool(1, 16, 1)
    k, v = grid_rows(rng, 2), grid_rows(rng, 2)
    oracle.quantize_append(pool, to_bf16_bits(k), to_bf16_bits(v), np.array([0, 1], dtype=np.int64))
    qb = to_bf16_bits(rng.standard_normal((1, 1, 128)) * 0.2)
    q = bf16_bits_to_f64(qb)[0, 0]
    out = oracle.decode_attention(pool, qb, np.zeros((1, 1), dtype=np.int32), np.array([2], dtype=np.int32), SM)
    d = SM * (q @ k[0] - q @ k[1])
    w0 = 1.0 / (1.0 + math.exp(-d))
    np.testing.assert_allclose(out[0, 0], w0 * v[0] + (1 - w0) * v[1], rtol=1e-12, atol=1e-12)


def test_empty_sequence_gives_zeros_and_placement_does_not_matter():
    rng = np.random.default_rng(10)
    lens = [0, 45, 100]
    pool, bt, ks, vs = build_cache(rng, lens, 2, 16, grid=False)
    q = to_bf16_bits(rng.standard_normal((3, 4, 128)))
    out = oracle.decode_attention(pool, q, bt, np.array(lens, dtype=np.int32), SM)
    assert not out[0].any()
    # move every page to a new physical place; results must be bit-identical
    perm = rng.permutation(pool.num_pages)
    pool2 = oracle.OraclePool(pool.num_pages, 16, 2)
    pool2.data[perm] = pool.data
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2 = oracle.decode_attention(pool2, q, bt2, np.array(lens, dtype=np.int32), SM)
    assert np.array_equal(out, out2)


def test_sequence_attention_agrees_with_paged_attention():
    rng = np.random.default_rng(11)
    lens = [77]
    pool, bt, ks, vs = build_cache(rng, lens, 2, 16, grid=False)
    q = to_bf16_bits(rng.standard_normal((1, 10, 128)))
    out = oracle.decode_attention(pool, q, bt, np.array(lens, dtype=np.int32), SM)
    for kv in range(2):
        o = oracle.sequence_attention(q[0, kv * 5:(kv + 1) * 5], to_bf16_bits(ks[0][:, kv]),
                                      to_bf16_bits(vs[0][:, kv]), SM)
        assert np.array_equal(o, out[0, kv * 5:(kv + 1) * 5])
        # rows wider than one head (the head's 128 values at each row start)
        kr = to_bf16_bits(ks[0].reshape(lens[0], -1))[:, kv * 128:]
        vr = to_bf16_bits(vs[0].reshape(lens[0], -1))[:, kv * 128:]
        o = oracle.sequence_attention(q[0, kv * 5:(kv + 1) * 5], kr, vr, SM)
        assert np.array_equal(o, out[0, kv * 5:(kv + 1) * 5])


def test_fp8_cache_attention_equals_sdpa_on_e4m3_values():
    rng = np.random.default_rng(12)
    lens = [40, 19]
    Hkv, P = 2, 16
    pool = oracle.OraclePool(8, P, Hkv, dtype=oracle.DTYPE_FP8)
    bt = np.array([[0, 5, 2], [7, 1, -1]], dtype=np.int32)
    ks, vs = [], []
    for b, n in enumerate(lens):
        k = torch.randn(n, Hkv, 128, dtype=torch.float64, generator=torch.Generator().manual_seed(b))
        v = torch.randn(n, Hkv, 128, dtype=torch.float64, generator=torch.Generator().manual_seed(b + 9))
        # values already on the E4M3 grid survive the FP8 cache exactly
        k = k.to(torch.float8_e4m3fn).to(torch.float64).numpy()
        v = v.to(torch.float8_e4m3fn).to(torch.float64).numpy()
        t = np.arange(n)
        oracle.quantize_append(pool, to_bf16_bits(k), to_bf16_bits(v), bt[b, t // P].astype(np.int64) * P + t % P)
        ks.append(k)
        vs.append(v)
    q_bits = to_bf16_bits(rng.standard_normal((2, 6, 128)))
    out = oracle.decode_attention(pool, q_bits, bt, np.array(lens, dtype=np.int32), SM)
    qf = torch.from_numpy(bf16_bits_to_f64(q_bits))
    for b in range(2):
        ref = F.scaled_dot_product_attention(qf[b][None, :, None], torch.from_numpy(ks[b]).permute(1, 0, 2)[None],
                                             torch.from_numpy(vs[b]).permute(1, 0, 2)[None], scale=SM,
                                             enable_gqa=True)[0, :, 0]
        np.testing.assert_allclose(out[b], ref.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("dtype", [oracle.DTYPE_NVFP4, oracle.DTYPE_FP8])
def test_prefix_dequant_round_trips_grid_values(dtype):
    rng = np.random.default_rng(13)
    lens = [0, 33, 64, 5]
    Hkv, P = 2, 16
    pool, bt, ks, vs = build_cache(rng, lens, Hkv, P, dtype=dtype, grid=(dtype == oracle.DTYPE_NVFP4))
    if dtype == oracle.DTYPE_FP8:  # make the reference the E4M3-rounded inputs
        ks = [torch.from_numpy(k.astype(np.float32)).to(torch.float8_e4m3fn).double().numpy() for k in ks]
        vs = [torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).double().numpy() for v in vs]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    kw, vw = oracle.prefix_dequant(pool, bt, np.array(lens, dtype=np.int32), cu)
    assert kw.shape == (sum(lens), Hkv, 128)
    for r, n in enumerate(lens):
        assert np.array_equal(bf16_bits_to_f64(kw[cu[r]:cu[r] + n]), ks[r])
        assert np.array_equal(bf16_bits_to_f64(vw[cu[r]:cu[r] + n]), vs[r])


@pytest.mark.parametrize("q_gain", [1.0, 300.0, 3.0e4])
def test_attention_agrees_with_extended_precision_over_wide_score_ranges(q_gain):
    """Scores up to ~1e7 (q scaled before BF16 rounding): the fp64 oracle must
    equal a brute-force softmax in extended precision (numpy longdouble,
    max-shifted) over the same lossless K/V; an unshifted exponential would
    overflow here."""
    if np.finfo(np.longdouble).eps >= np.finfo(np.float64).eps:
        pytest.skip("no extended precision on this host")
    rng = np.random.default_rng(int(q_gain) + 7)
    lens, Hq, Hkv, P = [45, 130], 8, 2, 16
    pool, bt, ks, vs = build_cache(rng, lens, Hkv, P)
    q_bits = to_bf16_bits(rng.standard_normal((len(lens), Hq, 128)) * q_gain)
    out = oracle.decode_attention(pool, q_bits, bt, np.array(lens, dtype=np.int32), SM, nthreads=2)
    q = bf16_bits_to_f64(q_bits).astype(np.longdouble)
    G = Hq // Hkv
    for b, n in enumerate(lens):
        k = ks[b].astype(np.longdouble)
        v = vs[b].astype(np.longdouble)
        for h in range(Hq):
            kv = h // G
            s = (k[:, kv, :] @ q[b, h]) * np.longdouble(SM)
            p = np.exp(s - s.max())
            ref = (p[:, None] * v[:, kv, :]).sum(axis=0) / p.sum()
            np.testing.assert_allclose(out[b, h], ref.astype(np.float64), rtol=1e-11, atol=1e-11 * float(np.abs(ref).max()))


def test_spread_closed_forms_and_sdpa_weights():
    """spread[h][d] = sum_t w_t |v_t[d] - out[h][d]|: zero for one token; half the
    gap for two tokens under equal weights; and, on grid values, the same sum
    formed from torch's float64 softmax weights (a library routine)."""
    rng = np.random.default_rng(21)
    pool, bt, ks, vs = build_cache(rng, [1, 2, 37], 1, 16)
    q = to_bf16_bits(rng.standard_normal((3, 2, 128)))
    lens = np.array([1, 2, 37], dtype=np.int32)
    out, spread = oracle.decode_attention(pool, q, bt, lens, SM, spread=True)
    assert np.array_equal(out, oracle.decode_attention(pool, q, bt, lens, SM))   # the output is unchanged
    assert not spread[0].any()
    qf = torch.from_numpy(bf16_bits_to_f64(q))
    for b, n in ((1, 2), (2, 37)):
        k = torch.from_numpy(ks[b][:, 0])
        v = torch.from_numpy(vs[b][:, 0])
        wts = torch.softmax(qf[b] @ k.T * SM, dim=-1)                       # [2][n]
        want = (wts[:, :, None] * (v[None] - torch.from_numpy(out[b])[:, None]).abs()).sum(1)
        np.testing.assert_allclose(spread[b], want.numpy(), rtol=1e-12, atol=1e-14)
    # identical keys: equal weights, spread = |v0 - v1| / 2
    pool2 = oracle.OraclePool(1, 16, 1)
    k = grid_rows(rng, 1).reshape(1, 128).repeat(2, 0)
    v = grid_rows(rng, 2).reshape(2, 128)
    oracle.quantize_append(pool2, to_bf16_bits(k), to_bf16_bits(v), np.arange(2, dtype=np.int64))
    _, s2 = oracle.decode_attention(pool2, q[:1, :1], np.zeros((1, 1), np.int32), np.array([2], np.int32), SM,
                                    spread=True)
    assert np.array_equal(s2[0, 0], np.abs(v[0] - v[1]) / 2)


def test_spread_of_sequence_and_extend_attention_match_decode():
    """The same spread from the oracle's three attention entry points on one sequence."""
    rng = np.random.default_rng(22)
    n = 45
    k = grid_rows(rng, n).reshape(n, 128)
    v = grid_rows(rng, n).reshape(n, 128)
    q = to_bf16_bits(rng.standard_normal((1, 4, 128)))
    pool = oracle.OraclePool(3, 16, 1)
    oracle.quantize_append(pool, to_bf16_bits(k), to_bf16_bits(v), np.arange(n, dtype=np.int64))
    o1, s1 = oracle.decode_attention(pool, q, np.arange(3, dtype=np.int32)[None], np.array([n], np.int32), SM,
                                     spread=True)
    o2, s2 = oracle.sequence_attention(q[0], to_bf16_bits(k), to_bf16_bits(v), SM, spread=True)
    kb, vb = to_bf16_bits(k).reshape(n, 1, 128), to_bf16_bits(v).reshape(n, 1, 128)
    o3, s3 = oracle.extend_attention(q, kb[:n - 1], vb[:n - 1], np.array([0, n - 1], np.int32), kb[n - 1:],
                                     vb[n - 1:], np.array([0, 1], np.int32), SM, spread=True)
    assert np.array_equal(o1[0], o2) and np.array_equal(s1[0], s2)
    np.testing.assert_allclose(o3[0], o2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(s3[0], s2, rtol=1e-12, atol=1e-13)
