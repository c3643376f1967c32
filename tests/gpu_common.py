"""Helpers for the GPU parity tests: build the same cache on the GPU (product
path) and in the oracle from the same BF16 bits, and the attention tolerance.

Tolerance of attention against the fp64 oracle, per element:

    |gpu - ref| <= max(2e-2, ulp_bf16(|ref| + eta) / 2 + eta),
    eta = (eps + 2^-16) * spread + 2^-16 * |ref|,

and relative L2 <= 3e-3 over the whole output.  spread = sum_t w_t |v_t - ref|
comes from the oracle (w_t its fp64 softmax weights).  The terms above 2e-2
are what the arithmetic forces, not a fit:

  * the output is BF16: the nearest BF16 number to a real lies up to half a
    BF16 step away (2^-6 in [4, 8), 2^-5 in [8, 16)), and the step is taken at
    |ref| + eta, where the kernel's FP32 result may lie;
  * eps is the relative rounding unit of the probabilities the kernel feeds to
    its P.V product -- 2^-11 where P is FP16 (decode, cascade), 2^-9 where it
    is BF16 (extend, as the page's BF16 BMM).  The same rounded P forms the
    numerator and the denominator, so the output is an exact average of the
    values under weights each off by a relative <= eps; since sum_t w_t
    (v_t - ref) = 0, that moves it by at most eps * spread (first order);
  * 2^-16 bounds the FP32 accumulations (24-bit sums over at most 2^8
    blocked partials per value) relative to sum_t w_t |v_t| <= spread + |ref|.

Where the values cluster around the output (spread small, the common case)
the bar is 2e-2 below |ref| = 8 and half a BF16 step just above it; it grows
past 2e-2 at small |ref| only when the weights sit on values far from the
output (outlier tokens), by eps * spread.
"""

import os

import numpy as np
import torch

import oracle

MAX_ABS = 2e-2
REL_L2 = 3e-3
EPS_FP16_P = 2.0**-11
EPS_BF16_P = 2.0**-9
FP32_REL = 2.0**-16


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of BF16 numbers at |x| (8 significant bits): 2^(floor(log2|x|) - 7)."""
    ax = np.maximum(np.abs(x), 2.0**-126)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def attention_bound(ref: np.ndarray, spread: np.ndarray, eps: float = EPS_FP16_P,
                    both_rounded: bool = False) -> np.ndarray:
    """Per-element bar for a BF16 output against ref (see the module doc).
    both_rounded: ref is itself another kernel's BF16 output, so each side is
    within half a step and eta of the exact value: a full step plus 2 eta."""
    a = np.abs(ref)
    eta = (eps + FP32_REL) * np.abs(spread) + FP32_REL * a
    if both_rounded:
        return np.maximum(MAX_ABS, bf16_ulp(a + 2 * eta) + 2 * eta)
    return np.maximum(MAX_ABS, 0.5 * bf16_ulp(a + eta) + eta)


def bits(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor -> numpy uint16 bit patterns (on the host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def check_attention(gpu_out, ref: np.ndarray, what: str = "", eps: float = EPS_FP16_P, spread=None,
                    both_rounded: bool = False):
    """Asserts the tolerance above (spread: the oracle's, same shape as ref);
    returns (max-abs error, rel-L2, the worst element's error / bound, ref
    there).  NVFP4KV_TOL_REPORT=1 prints one line per check."""
    if spread is None:
        raise TypeError("check_attention needs the oracle's spread")
    got = gpu_out.detach().float().cpu().double().numpy() if isinstance(gpu_out, torch.Tensor) else \
        np.asarray(gpu_out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    spread = np.broadcast_to(np.asarray(spread, dtype=np.float64), ref.shape)
    assert got.shape == ref.shape, "%s shape %s vs %s" % (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), "non-finite output " + what
    err = np.abs(got - ref)
    bound = attention_bound(ref, spread, eps, both_rounded)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref)) / denom if denom > 0 else float(np.linalg.norm(got - ref))
    ratio, ref_w = 0.0, 0.0
    if err.size:
        w = np.unravel_index(int(np.argmax(err / bound)), err.shape)
        ratio, ref_w = float(err[w] / bound[w]), float(ref[w])
        if os.environ.get("NVFP4KV_TOL_REPORT"):
            a = np.unravel_index(int(np.argmax(err)), err.shape)
            print("\nTOL %s: worst err/bound %.3f (err %.3e, bound %.3e, ref %.6g, spread %.4g); max-abs %.3e at "
                  "ref %.6g; bar above 2e-2 on %.2f%% of elements; rel-L2 %.3e"
                  % (what, ratio, err[w], bound[w], ref[w], spread[w], max_abs, ref[a],
                     100.0 * float(np.mean(bound > MAX_ABS)), rel))
        assert err[w] <= bound[w], "%s |err| %.3e > bound %.3e at %s (ref %.6g, got %.6g, spread %.4g)" % (
            what, err[w], bound[w], w, ref[w], got[w], spread[w])
    assert rel <= REL_L2, "%s rel-L2 %.3e > %.1e" % (what, rel, REL_L2)
    return max_abs, rel, ratio, ref_w


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
    ref, spread = oracle.decode_attention(pool, bits(q), w.block_table.numpy(), w.seq_lens.numpy(), w.sm_scale,
                                          spread=True)
    return out, ref, spread
