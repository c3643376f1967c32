"""CPU oracle for the NVFP4 paged KV cache -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The product package
(``nvfp4_quantised_paged_gb300``) never imports it and shares no code with it.

Everything here is a thin numpy/ctypes wrapper around ``nvfp4kv_oracle.c``,
which holds the arithmetic (see its header for what is computed, the page and
section each step follows, and the readings taken where the page is silent).

Arrays crossing the boundary:
  BF16 tensors are passed as ``numpy.uint16`` bit patterns; the pool is a
  ``numpy.uint8`` array laid out as in the C file; outputs are ``float64``
  (attention) or ``uint16`` BF16 bits (prefix dequant).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4kv_oracle.c")
_LIB = os.path.join(_HERE, "libnvfp4kv_oracle.so")

DTYPE_NVFP4 = 0
DTYPE_FP8 = 1
HEAD_DIM = 128

OK, EINVAL, ENONFINITE, ESLOT, EPAGE = 0, -1, -2, -3, -4

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no GPU, no CUDA); returns the .so path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-shared", "-fPIC",
               "-pthread", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f32, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
        sig = {
            "oracle_calibrate_global_scale": (f32, [P, i64]),
            "oracle_extend_attention": (i32, [P, P, P, P, P, P, P, i32, i32, i32, f64, P, P, i32]),
            "oracle_bf16_value": (f64, [ctypes.c_uint16]),
            "oracle_bf16_from_float": (ctypes.c_uint16, [f32]),
            "oracle_bf16_from_double": (ctypes.c_uint16, [f64]),
            "oracle_e4m3_value": (f64, [ctypes.c_uint8]),
            "oracle_e2m1_value": (f64, [ctypes.c_uint8]),
            "oracle_e4m3_encode": (ctypes.c_uint8, [f32]),
            "oracle_e2m1_encode": (ctypes.c_uint8, [f32]),
            "oracle_e2m1_encode_quotients": (None, [P, P, i64, P]),
            "oracle_e4m3_encode_many": (None, [P, i64, P]),
            "oracle_quantize_block16": (i32, [P, f32, P, P]),
            "oracle_slab_bytes": (i64, [i32, i32]),
            "oracle_quantize_append": (i32, [P, i64, i32, i32, i32, f32, f32, P, P, i64, i64, P]),
            "oracle_decode_attention": (i32, [P, i64, i32, i32, i32, f32, f32, P, i32, i32, P, i32, P, f64,
                                              P, P, i32]),
            "oracle_sequence_attention": (i32, [P, i32, P, P, i64, i64, i32, f32, f32, f64, P, P]),
            "oracle_prefix_dequant": (i32, [P, i64, i32, i32, i32, f32, f32, P, i32, P, P, i32, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _check(rc: int, what: str):
    if rc != OK:
        raise ValueError("oracle %s failed with status %d" % (what, rc))


class OraclePool:
    """A host page pool with the cache's layout (uint8[num_pages][Hkv][slab])."""

    def __init__(self, num_pages, page_size, num_kv_heads, dtype=DTYPE_NVFP4, gk=1.0, gv=1.0, fill=0):
        self.num_pages, self.page_size, self.num_kv_heads = int(num_pages), int(page_size), int(num_kv_heads)
        self.dtype, self.gk, self.gv = int(dtype), float(gk), float(gv)
        self.slab = int(slab_bytes(self.dtype, self.page_size))
        self.data = np.full((self.num_pages, self.num_kv_heads, self.slab), fill, dtype=np.uint8)

    def _hdr(self):
        return (_ptr(self.data), self.num_pages, self.page_size, self.num_kv_heads, self.dtype, self.gk, self.gv)


# ---------------------------------------------------------------- scalar codecs

def bf16_value(bits: int) -> float:
    return _load().oracle_bf16_value(int(bits))


def bf16_from_double(x: float) -> int:
    """BF16 bits of x rounded once, nearest-even (subnormals, overflow to infinity)."""
    return int(_load().oracle_bf16_from_double(float(x)))


def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(int(code))


def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(int(code))


def e4m3_encode(x: float) -> int:
    return int(_load().oracle_e4m3_encode(float(x)))


def e2m1_encode(x: float) -> int:
    return int(_load().oracle_e2m1_encode(float(x)))


def e4m3_encode_many(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_many(_ptr(x), x.size, _ptr(out))
    return out


def e2m1_encode_quotients(x: np.ndarray, d: np.ndarray) -> np.ndarray:
    """code_i = E2M1(fl32(x_i / d_i)) for float32 arrays of one shape."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    d = np.ascontiguousarray(np.broadcast_to(d, x.shape), dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_e2m1_encode_quotients(_ptr(x), _ptr(d), x.size, _ptr(out))
    return out


def quantize_block16(x_bf16: np.ndarray, g: float = 1.0):
    """Returns (codes[16] one per byte, scale_code) for 16 BF16 bit patterns."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(16)
    codes = np.zeros(16, dtype=np.uint8)
    scale = np.zeros(1, dtype=np.uint8)
    _check(_load().oracle_quantize_block16(_ptr(x), float(g), _ptr(codes), _ptr(scale)), "quantize_block16")
    return codes, int(scale[0])


def calibrate_global_scale(x_bf16: np.ndarray) -> np.float32:
    """FP32 tensor scale g = amax / (6 * 448) over the finite BF16 values (bits)
    of x; 1.0 for an all-zero tensor."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(-1)
    return np.float32(_load().oracle_calibrate_global_scale(_ptr(x), x.size))


def slab_bytes(dtype: int, page_size: int) -> int:
    return int(_load().oracle_slab_bytes(int(dtype), int(page_size)))


# ---------------------------------------------------------------- the three paths

def quantize_append(pool: OraclePool, k: np.ndarray, v: np.ndarray, slot_mapping: np.ndarray):
    """k, v: uint16 BF16 bits [T][Hkv*128] (or [T][Hkv][128]); slot_mapping int64 [T]."""
    T = int(slot_mapping.shape[0])
    if T == 0:
        return
    k = np.ascontiguousarray(k, dtype=np.uint16).reshape(T, -1)
    v = np.ascontiguousarray(v, dtype=np.uint16).reshape(T, -1)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    rc = _load().oracle_quantize_append(*pool._hdr(), _ptr(k), _ptr(v), T, k.shape[1], _ptr(sm))
    _check(rc, "quantize_append")


def _spread_arg(spread: bool, out: np.ndarray):
    sp = np.zeros_like(out) if spread else None
    return sp, (_ptr(sp) if spread else None)


def decode_attention(pool: OraclePool, q: np.ndarray, block_table: np.ndarray, seq_lens: np.ndarray,
                     sm_scale: float, nthreads: int = 0, spread: bool = False):
    """q: uint16 BF16 bits [B][Hq][128]; returns float64 [B][Hq][128], or with
    spread=True (out, spread): spread[b][h][d] = sum_t w_t |v_t[d] - out[b][h][d]|
    over the softmax weights w_t (the error scale the parity tests use)."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    B, Hq = int(q.shape[0]), int(q.shape[1])
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((B, Hq, HEAD_DIM), dtype=np.float64)
    sp, sp_ptr = _spread_arg(spread, out)
    rc = _load().oracle_decode_attention(*pool._hdr(), _ptr(q), B, Hq, _ptr(bt), bt.shape[1], _ptr(sl),
                                         float(sm_scale), _ptr(out), sp_ptr, int(nthreads))
    _check(rc, "decode_attention")
    return (out, sp) if spread else out


def sequence_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float, dtype: int = DTYPE_NVFP4,
                       gk: float = 1.0, gv: float = 1.0, spread: bool = False):
    """Attention of G query heads over one sequence given as BF16 K/V rows.

    q: uint16 [G][128]; k, v: uint16 [n][128] (one KV head).  Returns float64
    [G][128], or (out, spread) as decode_attention does.
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    G, n = int(q.shape[0]), int(k.shape[0])
    out = np.zeros((G, HEAD_DIM), dtype=np.float64)
    sp, sp_ptr = _spread_arg(spread, out)
    rc = _load().oracle_sequence_attention(_ptr(q), G, _ptr(k), _ptr(v), n, k.shape[1], int(dtype), float(gk),
                                           float(gv), float(sm_scale), _ptr(out), sp_ptr)
    _check(rc, "sequence_attention")
    return (out, sp) if spread else out


def prefix_dequant(pool: OraclePool, block_table: np.ndarray, prefix_lens: np.ndarray,
                   cu_prefix_lens: np.ndarray):
    """Returns (k_ws, v_ws) uint16 BF16 bits [total][Hkv][128]."""
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    pl = np.ascontiguousarray(prefix_lens, dtype=np.int32)
    cu = np.ascontiguousarray(cu_prefix_lens, dtype=np.int32)
    total = int(cu[-1]) if cu.size else 0
    k_ws = np.zeros((total, pool.num_kv_heads, HEAD_DIM), dtype=np.uint16)
    v_ws = np.zeros((total, pool.num_kv_heads, HEAD_DIM), dtype=np.uint16)
    rc = _load().oracle_prefix_dequant(*pool._hdr(), _ptr(bt), bt.shape[1], _ptr(pl), _ptr(cu), int(pl.shape[0]),
                                       _ptr(k_ws), _ptr(v_ws))
    _check(rc, "prefix_dequant")
    return k_ws, v_ws


# ---------------------------------------------------------------- BF16 helpers

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact BF16 bits -> float64 (a bit shift, no rounding)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def extend_attention(q: np.ndarray, k_prefix: np.ndarray, v_prefix: np.ndarray, cu_prefix: np.ndarray,
                     k_chunk: np.ndarray, v_chunk: np.ndarray, cu_q: np.ndarray, sm_scale: float,
                     nthreads: int = 0, spread: bool = False):
    """fp64 extend attention: chunk token i of request r attends to its prefix
    rows (BF16 bits [total_prefix][Hkv][128], rows cu_prefix[r]..cu_prefix[r+1])
    and to chunk tokens 0..i (BF16 bits [total_q][Hkv][128]); q: BF16 bits
    [total_q][Hq][128].  Returns float64 [total_q][Hq][128], or (out, spread) as
    decode_attention does."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kp, vp = np.ascontiguousarray(k_prefix, dtype=np.uint16), np.ascontiguousarray(v_prefix, dtype=np.uint16)
    kn, vn = np.ascontiguousarray(k_chunk, dtype=np.uint16), np.ascontiguousarray(v_chunk, dtype=np.uint16)
    cp = np.ascontiguousarray(cu_prefix, dtype=np.int32)
    cq = np.ascontiguousarray(cu_q, dtype=np.int32)
    total_q, hq = q.shape[0], q.shape[1]
    hkv = kn.shape[1] if kn.ndim == 3 else kp.shape[1]
    out = np.zeros((total_q, hq, HEAD_DIM), dtype=np.float64)
    # a valid (never dereferenced) pointer for empty arrays
    kp = kp if kp.size else np.zeros(1, np.uint16)
    vp = vp if vp.size else np.zeros(1, np.uint16)
    sp, sp_ptr = _spread_arg(spread, out)
    rc = _load().oracle_extend_attention(_ptr(q), _ptr(kp), _ptr(vp), _ptr(cp), _ptr(kn), _ptr(vn), _ptr(cq),
                                         len(cq) - 1, hq, hkv, float(sm_scale), _ptr(out), sp_ptr, int(nthreads))
    _check(rc, "extend_attention")
    return (out, sp) if spread else out
