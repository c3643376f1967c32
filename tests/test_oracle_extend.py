"""Pins of the oracle's extend attention (section A2, path 2: the chunk attends
to [cached prefix as the BF16 workspace holds it || its own K/V], causally
within the chunk): torch's scaled_dot_product_attention in float64 with the
prefix-plus-causal mask, the pure causal case (no prefix), and the link to
path 3 -- a one-token chunk over a prefix read back from the NVFP4 pool is
the decode attention of that pool with the token appended."""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle_helpers import bf16_bits_to_f64, grid_rows, to_bf16_bits

SM = 1.0 / math.sqrt(128)


def _sdpa_ref(q, kp, vp, kn, vn, cu_p, cu_q):
    """float64 SDPA per request with mask[i, t] = t < n_prefix + i + 1."""
    out = np.zeros(q.shape, dtype=np.float64)
    qf, kpf, vpf = bf16_bits_to_f64(q), bf16_bits_to_f64(kp), bf16_bits_to_f64(vp)
    knf, vnf = bf16_bits_to_f64(kn), bf16_bits_to_f64(vn)
    for r in range(len(cu_q) - 1):
        a, b = cu_q[r], cu_q[r + 1]
        pa, pb = cu_p[r], cu_p[r + 1]
        L, npre = b - a, pb - pa
        if L == 0:
            continue
        k = np.concatenate([kpf[pa:pb], knf[a:b]])          # [n][Hkv][D]
        v = np.concatenate([vpf[pa:pb], vnf[a:b]])
        mask = np.arange(npre + L)[None, :] < (npre + np.arange(L) + 1)[:, None]
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(qf[a:b]).permute(1, 0, 2)[None], torch.from_numpy(k).permute(1, 0, 2)[None],
            torch.from_numpy(v).permute(1, 0, 2)[None], attn_mask=torch.from_numpy(mask), scale=SM, enable_gqa=True)
        out[a:b] = ref[0].permute(1, 0, 2).numpy()
    return out


def _inputs(rng, prefix_lens, chunk_lens, Hq, Hkv):
    cu_p = np.concatenate([[0], np.cumsum(prefix_lens)]).astype(np.int32)
    cu_q = np.concatenate([[0], np.cumsum(chunk_lens)]).astype(np.int32)
    bf = lambda *s: to_bf16_bits(rng.standard_normal(s))
    return (bf(cu_q[-1], Hq, 128), bf(cu_p[-1], Hkv, 128), bf(cu_p[-1], Hkv, 128), bf(cu_q[-1], Hkv, 128),
            bf(cu_q[-1], Hkv, 128), cu_p, cu_q)


@pytest.mark.parametrize("prefix_lens,chunk_lens,Hq,Hkv", [
    ([40, 0, 130], [7, 20, 33], 8, 2),
    ([300], [64], 32, 8),
    ([5, 17], [1, 0], 5, 1),
])
def test_extend_equals_sdpa_with_prefix_causal_mask(prefix_lens, chunk_lens, Hq, Hkv):
    rng = np.random.default_rng(sum(prefix_lens) + sum(chunk_lens) + Hq)
    q, kp, vp, kn, vn, cu_p, cu_q = _inputs(rng, prefix_lens, chunk_lens, Hq, Hkv)
    got = oracle.extend_attention(q, kp, vp, cu_p, kn, vn, cu_q, SM, nthreads=4)
    np.testing.assert_allclose(got, _sdpa_ref(q, kp, vp, kn, vn, cu_p, cu_q), rtol=1e-12, atol=1e-12)


def test_no_prefix_is_plain_causal_attention():
    rng = np.random.default_rng(3)
    q, kp, vp, kn, vn, cu_p, cu_q = _inputs(rng, [0], [50], 4, 4)
    got = oracle.extend_attention(q, kp, vp, cu_p, kn, vn, cu_q, SM)
    ref = F.scaled_dot_product_attention(*(torch.from_numpy(bf16_bits_to_f64(x)).permute(1, 0, 2)[None]
                                           for x in (q, kn, vn)), is_causal=True, scale=SM)
    np.testing.assert_allclose(got, ref[0].permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)
    # the first chunk token sees only itself: its output is its own value row
    np.testing.assert_array_equal(got[0], bf16_bits_to_f64(vn[0]))


def test_one_token_chunk_over_a_cached_prefix_is_decode_attention():
    rng = np.random.default_rng(4)
    P, Hkv, Hq, n = 16, 2, 8, 37
    # prefix and the new token are grid-valued, so the pool stores them losslessly
    k = grid_rows(rng, (n + 1) * Hkv).reshape(n + 1, Hkv, 128)
    v = grid_rows(rng, (n + 1) * Hkv).reshape(n + 1, Hkv, 128)
    pages = -(-(n + 1) // P)
    pool = oracle.OraclePool(pages + 2, P, Hkv)
    bt = rng.permutation(pages + 2)[:pages].astype(np.int32)[None]
    t = np.arange(n + 1)
    oracle.quantize_append(pool, to_bf16_bits(k), to_bf16_bits(v), bt[0, t // P].astype(np.int64) * P + t % P)
    q = to_bf16_bits(rng.standard_normal((1, Hq, 128)))
    dec = oracle.decode_attention(pool, q, bt, np.array([n + 1], np.int32), SM)
    kp, vp = oracle.prefix_dequant(pool, bt, np.array([n], np.int32), np.array([0, n], np.int32))
    ext = oracle.extend_attention(q, kp, vp, np.array([0, n], np.int32), to_bf16_bits(k[n:]), to_bf16_bits(v[n:]),
                                  np.array([0, 1], np.int32), SM)
    np.testing.assert_allclose(ext, dec, rtol=1e-13, atol=1e-13)
