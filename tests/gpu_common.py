"""Helpers for the GPU parity tests: build the same cache on the GPU (product
path) and in the oracle from the same BF16 bits, and the attention tolerance.

Tolerance of decode attention against the fp64 oracle: per element
|gpu - ref| <= max(2e-2, ulp_bf16(ref)), and relative L2 <= 3e-3 over the
whole output.  The output is BF16, whose spacing exceeds 2e-2 once
|ref| >= 4 (an element in [8, 16) cannot be stored closer than 2^-5 to an
arbitrary real), so above that the bar is one BF16 step; below |ref| = 4 it
is exactly 2e-2.
"""

import numpy as np
import torch

import oracle

MAX_ABS = 2e-2
REL_L2 = 3e-3


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of BF16 numbers at |x| (8 significant bits): 2^(floor(log2|x|) - 7)."""
    ax = np.maximum(np.abs(x), 2.0**-126)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def bits(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor -> numpy uint16 bit patterns (on the host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def check_attention(gpu_out: torch.Tensor, ref: np.ndarray, what: str = ""):
    got = gpu_out.detach().float().cpu().double().numpy()
    assert np.isfinite(got).all(), "non-finite output " + what
    err = np.abs(got - ref)
    bound = np.maximum(MAX_ABS, bf16_ulp(ref))
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref)) / denom if denom > 0 else float(np.linalg.norm(got - ref))
    if err.size:
        w = np.unravel_index(int(np.argmax(err / bound)), err.shape)
        assert err[w] <= bound[w], "%s |err| %.3e > bound %.3e at %s (ref %.6g, got %.6g)" % (
            what, err[w], bound[w], w, ref[w], got[w])
    assert rel <= REL_L2, "%s rel-L2 %.3e > %.1e" % (what, rel, REL_L2)
    return max_abs, rel


def fill_both(w, m, dtype=0, gk=1.0, gv=1.0, device="cuda"):
    """Quantise-append every sequence of DecodeWorkload w into a GPU cache and an
    oracle pool; returns (gpu cache, oracle pool)."""
    cache = m.PagedCache(w.num_pages, w.page_size, w.num_kv_heads, dtype=dtype, k_global_scale=gk,
                         v_global_scale=gv, device=device)
    pool = oracle.OraclePool(w.num_pages, w.page_size, w.num_kv_heads, dtype=dtype, gk=gk, gv=gv)
    if w.shared_prefix_tokens:
        pk, pv = w.prefix_kv(device)
        slots = w.slots(0, 0, w.shared_prefix_tokens)
        m.quantize_append(cache, pk, pv, slots.to(device))
        oracle.quantize_append(pool, bits(pk), bits(pv), slots.numpy())
    for b in range(w.batch):
        k, v = w.private_kv(b, device)
        if k.shape[0] == 0:
            continue
        slots = w.slots(b, w.shared_prefix_tokens)
        m.quantize_append(cache, k, v, slots.to(device))
        oracle.quantize_append(pool, bits(k), bits(v), slots.numpy())
    torch.cuda.synchronize()
    return cache, pool


def decode_both(w, m, cache, pool, num_splits=0, device="cuda"):
    q = w.q(device)
    bt = w.block_table.to(device)
    sl = w.seq_lens.to(device)
    out = m.paged_decode_attention(cache, q, bt, sl, w.sm_scale, num_splits=num_splits)
    torch.cuda.synchronize()
    assert m.check_device_errors() == 0
    ref = oracle.decode_attention(pool, bits(q), w.block_table.numpy(), w.seq_lens.numpy(), w.sm_scale)
    return out, ref
