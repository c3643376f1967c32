"""Python binding of libnvfp4kv.so, the NVFP4 paged KV cache library for GB300.

Argument marshalling only: every step of the cache paths runs in the CUDA
kernels behind the C ABI (include/nvfp4kv.h).  PyTorch provides device
memory and streams.  There is no CPU fallback: importing this package on a
machine without the built library, or calling it without a CUDA device,
raises.

The three paths of "Accelerating Long-Context and Agentic Inference with
NVFP4 KV Cache" (section A2):

  quantize_append(cache, k, v, slot_mapping)             paths 1 and 2 (write)
  paged_decode_attention(cache, q, block_table, seq_lens) path 3 (decode)
  prefix_dequant(cache, block_table, prefix_lens, cu)     path 2 (extend)
"""

from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libnvfp4kv.so")

DTYPE_NVFP4 = 0
DTYPE_FP8_E4M3 = 1
HEAD_DIM = 128

STATUS = {0: "ok", -1: "invalid argument", -2: "unsupported configuration", -3: "CUDA error",
          -4: "a kernel skipped an out-of-range index"}


class NVFP4KVError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s failed: %s (status %d)" % (what, STATUS.get(status, "unknown"), status))
        self.status = status


class _CacheDesc(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("num_pages", ctypes.c_int64), ("page_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("k_global_scale", ctypes.c_float), ("v_global_scale", ctypes.c_float)]


def _load_library():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libnvfp4kv.so is not built; run __graft_entry__.build() (nvcc, sm_103a) first: %s"
                          % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    D = ctypes.POINTER(_CacheDesc)
    sig = {
        "nvfp4kv_version": (i32, []),
        "nvfp4kv_status_string": (ctypes.c_char_p, [i32]),
        "nvfp4kv_slab_bytes": (sz, [D]),
        "nvfp4kv_pool_bytes": (sz, [D]),
        "nvfp4_kv_quantize_append": (i32, [D, P, P, i64, i64, P, P]),
        "nvfp4kv_decode_workspace_bytes": (sz, [D, i32, i32, i32]),
        "nvfp4kv_decode_auto_splits": (i32, [D, i32]),
        "nvfp4kv_decode_launch_count": (i32, [D, i32, i32, i32, i32]),
        "nvfp4_paged_decode_attention": (i32, [D, P, i32, i32, P, i32, P, f32, P, P, sz, i32, P]),
        "nvfp4_prefix_dequant": (i32, [D, P, i32, P, P, i32, i64, P, P, P]),
        "nvfp4kv_check_device_errors": (i32, [P]),
        "nvfp4kv_selftest_bounded_wait": (i32, [i32, ctypes.c_uint, P, P]),
        "nvfp4kv_calibrate_global_scales": (i32, [P, P, i64, i32, i64, P, P]),
        "nvfp4_extend_attention": (i32, [P, P, P, P, i64, P, P, P, i64, i32, i32, i32, i32, f32, P, P]),
        "nvfp4_extend_attention_paged": (i32, [D, P, P, i32, P, P, P, P, i64, i32, i32, i32, f32, P, P]),
        "nvfp4_paged_decode_attention_append": (i32, [D, P, P, i64, P, i32, i32, P, i32, P, f32, P, P, sz, i32, P]),
        "nvfp4kv_cascade_workspace_bytes": (sz, [D, i32, i32, i32, i32]),
        "nvfp4_cascade_decode_attention": (i32, [D, P, i32, i32, P, i32, P, i32, P, f32, P, P, sz, i32, P]),
        "nvfp4kv_profile_decode": (i32, [P, P, i32, i32]),
        "nvfp4_paged_decode_attention_noalloc": (i32, [D, P, i32, i32, P, i32, P, f32, P, i32, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load_library()

EXPORTED_SYMBOLS = ("nvfp4kv_version", "nvfp4kv_status_string", "nvfp4kv_slab_bytes", "nvfp4kv_pool_bytes",
                    "nvfp4_kv_quantize_append", "nvfp4kv_decode_workspace_bytes", "nvfp4kv_decode_auto_splits",
                    "nvfp4kv_decode_launch_count",
                    "nvfp4_paged_decode_attention", "nvfp4_prefix_dequant", "nvfp4kv_check_device_errors",
                    "nvfp4kv_profile_decode", "nvfp4_paged_decode_attention_noalloc",
                    "nvfp4kv_selftest_bounded_wait", "nvfp4kv_calibrate_global_scales", "nvfp4_extend_attention",
                    "nvfp4_extend_attention_paged",
                    "nvfp4_paged_decode_attention_append", "nvfp4kv_cascade_workspace_bytes",
                    "nvfp4_cascade_decode_attention")

NOALLOC_SCRATCH_BYTES = 64 << 20  # NVFP4KV_NOALLOC_SCRATCH_BYTES of the header


def library():
    """The loaded ctypes library (for tests of the raw ABI)."""
    return _lib


def _check(rc: int, what: str):
    if rc != 0:
        raise NVFP4KVError(rc, what)


def _stream(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr() if t is not None else 0)


def _require(t: torch.Tensor, name: str, dtype: torch.dtype):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


class PagedCache:
    """A caller-owned page pool (uint8 [num_pages][num_kv_heads][slab]) and its format."""

    def __init__(self, num_pages: int, page_size: int, num_kv_heads: int, dtype: int = DTYPE_NVFP4,
                 k_global_scale: float = 1.0, v_global_scale: float = 1.0, device="cuda",
                 pool: Optional[torch.Tensor] = None):
        self.num_pages, self.page_size, self.num_kv_heads = int(num_pages), int(page_size), int(num_kv_heads)
        self.dtype = int(dtype)
        self.k_global_scale, self.v_global_scale = float(k_global_scale), float(v_global_scale)
        slab = slab_bytes(self.dtype, self.page_size, self.num_kv_heads)
        self.slab = slab
        if pool is None:
            pool = torch.zeros((self.num_pages, self.num_kv_heads, slab), dtype=torch.uint8, device=device)
        _require(pool, "pool", torch.uint8)
        if pool.numel() != self.num_pages * self.num_kv_heads * slab:
            raise ValueError("pool has %d bytes, expected %d" % (pool.numel(), self.num_pages * self.num_kv_heads * slab))
        self.pool = pool
        self._desc = _CacheDesc(pool.data_ptr(), self.num_pages, self.page_size, self.num_kv_heads, HEAD_DIM,
                                self.dtype, self.k_global_scale, self.v_global_scale)

    @property
    def desc(self):
        return ctypes.byref(self._desc)

    @property
    def num_slots(self) -> int:
        return self.num_pages * self.page_size


def slab_bytes(dtype: int, page_size: int, num_kv_heads: int = 1) -> int:
    d = _CacheDesc(256, 1, page_size, num_kv_heads, HEAD_DIM, dtype, 1.0, 1.0)
    n = _lib.nvfp4kv_slab_bytes(ctypes.byref(d))
    if n == 0:
        raise NVFP4KVError(-2, "slab_bytes(dtype=%d, page_size=%d)" % (dtype, page_size))
    return int(n)


def quantize_append(cache: PagedCache, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                    stream: Optional[torch.cuda.Stream] = None):
    """k, v: BF16 [T][Hkv][128] or [T][stride >= Hkv*128]; slot_mapping: int64 [T]."""
    T = int(slot_mapping.shape[0])
    _require(slot_mapping, "slot_mapping", torch.int64)
    row = cache.num_kv_heads * HEAD_DIM
    for name, x in (("k", k), ("v", v)):
        if not x.is_cuda or x.dtype != torch.bfloat16:
            raise ValueError("%s must be a CUDA bfloat16 tensor" % name)
        if x.shape[0] != T:
            raise ValueError("%s has %d tokens, slot_mapping %d" % (name, x.shape[0], T))
        # each token's Hkv*128 values contiguous; tokens may be strided (a view of a wider QKV buffer)
        if T > 0 and (not x[0].is_contiguous() or x[0].numel() != row):
            raise ValueError("%s: each token must hold %d contiguous values" % (name, row))
    stride = int(k.stride(0)) if T > 0 else row
    if T > 0 and int(v.stride(0)) != stride:
        raise ValueError("k and v must share a token stride")
    rc = _lib.nvfp4_kv_quantize_append(cache.desc, _ptr(k), _ptr(v), T, stride, _ptr(slot_mapping), _stream(stream))
    _check(rc, "nvfp4_kv_quantize_append")


def calibrate_global_scales(k: torch.Tensor, v: torch.Tensor, num_kv_heads: int,
                            stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Per-tensor FP32 global scales {g_K, g_V} = amax / (6 * 448) of BF16 K and V
    ([T][Hkv][128] or token-strided, as for quantize_append), as a device float32
    tensor [2] (1.0 for an all-zero tensor)."""
    T = int(k.shape[0])
    row = int(num_kv_heads) * HEAD_DIM
    for name, x in (("k", k), ("v", v)):
        if not x.is_cuda or x.dtype != torch.bfloat16:
            raise ValueError("%s must be a CUDA bfloat16 tensor" % name)
        if x.shape[0] != T:
            raise ValueError("k and v must have the same number of tokens")
        if T > 0 and (not x[0].is_contiguous() or x[0].numel() != row):
            raise ValueError("%s: each token must hold %d contiguous values" % (name, row))
    stride = int(k.stride(0)) if T > 0 else row
    if T > 0 and int(v.stride(0)) != stride:
        raise ValueError("k and v must share a token stride")
    scales = torch.empty(2, dtype=torch.float32, device=k.device)
    rc = _lib.nvfp4kv_calibrate_global_scales(_ptr(k), _ptr(v), T, int(num_kv_heads), stride, _ptr(scales),
                                              _stream(stream))
    _check(rc, "nvfp4kv_calibrate_global_scales")
    return scales


def decode_workspace_bytes(cache: PagedCache, batch: int, num_q_heads: int, num_splits: int = 0) -> int:
    n = _lib.nvfp4kv_decode_workspace_bytes(cache.desc, int(batch), int(num_q_heads), int(num_splits))
    if n == 0 and batch > 0:
        raise NVFP4KVError(-1, "decode_workspace_bytes")
    return int(n)


def decode_auto_splits(cache: PagedCache, num_q_heads: int) -> int:
    return int(_lib.nvfp4kv_decode_auto_splits(cache.desc, int(num_q_heads)))


def decode_launch_count(cache: PagedCache, batch: int, num_q_heads: int, num_splits: int = 0,
                        shared_len: int = 0) -> int:
    """Kernel launches of one decode (shared_len = 0) or cascade call of this shape."""
    return int(_lib.nvfp4kv_decode_launch_count(cache.desc, int(batch), int(num_q_heads), int(num_splits),
                                                int(shared_len)))


def alloc_decode_workspace(cache: PagedCache, batch: int, num_q_heads: int, num_splits: int = 0) -> torch.Tensor:
    n = decode_workspace_bytes(cache, batch, num_q_heads, num_splits)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=cache.pool.device)


def paged_decode_attention(cache: PagedCache, q: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                           sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, num_splits: int = 0,
                           stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """q: BF16 [B][Hq][128]; block_table int32 [B][max_pages]; seq_lens int32 [B] -> BF16 [B][Hq][128]."""
    _require(q, "q", torch.bfloat16)
    _require(block_table, "block_table", torch.int32)
    _require(seq_lens, "seq_lens", torch.int32)
    B, Hq = int(q.shape[0]), int(q.shape[1])
    if q.shape[2] != HEAD_DIM:
        raise ValueError("head_dim must be 128")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    if out is None:
        out = torch.empty_like(q)
    _require(out, "out", torch.bfloat16)
    if workspace is None:
        workspace = alloc_decode_workspace(cache, B, Hq, num_splits)
    _require(workspace, "workspace", torch.uint8)
    rc = _lib.nvfp4_paged_decode_attention(cache.desc, _ptr(q), B, Hq, _ptr(block_table), int(block_table.shape[1]),
                                           _ptr(seq_lens), float(sm_scale), _ptr(out), _ptr(workspace),
                                           workspace.numel(), int(num_splits), _stream(stream))
    _check(rc, "nvfp4_paged_decode_attention")
    return out


def paged_decode_attention_append(cache: PagedCache, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
                                  block_table: torch.Tensor, seq_lens: torch.Tensor, sm_scale: Optional[float] = None,
                                  out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                                  num_splits: int = 0, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Decode step with the new token appended in the same launch: row b of
    k_new / v_new (BF16 [B][Hkv][128], or token-strided) is quantised into
    position seq_lens[b] - 1 of sequence b, then attention as paged_decode_attention."""
    _require(q, "q", torch.bfloat16)
    _require(block_table, "block_table", torch.int32)
    _require(seq_lens, "seq_lens", torch.int32)
    B, Hq = int(q.shape[0]), int(q.shape[1])
    if q.shape[2] != HEAD_DIM:
        raise ValueError("head_dim must be 128")
    row = cache.num_kv_heads * HEAD_DIM
    for name, x in (("k_new", k_new), ("v_new", v_new)):
        if not x.is_cuda or x.dtype != torch.bfloat16 or x.shape[0] != B:
            raise ValueError("%s must be a CUDA bfloat16 tensor with one row per sequence" % name)
        if B > 0 and (not x[0].is_contiguous() or x[0].numel() != row):
            raise ValueError("%s: each row must hold %d contiguous values" % (name, row))
    stride = int(k_new.stride(0)) if B > 0 else row
    if B > 0 and int(v_new.stride(0)) != stride:
        raise ValueError("k_new and v_new must share a row stride")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    if out is None:
        out = torch.empty_like(q)
    _require(out, "out", torch.bfloat16)
    if workspace is None:
        workspace = alloc_decode_workspace(cache, B, Hq, num_splits)
    _require(workspace, "workspace", torch.uint8)
    rc = _lib.nvfp4_paged_decode_attention_append(cache.desc, _ptr(k_new), _ptr(v_new), stride, _ptr(q), B, Hq,
                                                  _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
                                                  float(sm_scale), _ptr(out), _ptr(workspace), workspace.numel(),
                                                  int(num_splits), _stream(stream))
    _check(rc, "nvfp4_paged_decode_attention_append")
    return out


def cascade_workspace_bytes(cache: PagedCache, batch: int, num_q_heads: int, shared_len: int,
                            num_splits: int = 0) -> int:
    n = _lib.nvfp4kv_cascade_workspace_bytes(cache.desc, int(batch), int(num_q_heads), int(num_splits),
                                             int(shared_len))
    if n == 0 and batch > 0:
        raise NVFP4KVError(-1, "cascade_workspace_bytes")
    return int(n)


def cascade_decode_attention(cache: PagedCache, q: torch.Tensor, shared_pages: torch.Tensor, shared_len: int,
                             block_table: torch.Tensor, seq_lens: torch.Tensor, sm_scale: Optional[float] = None,
                             out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                             num_splits: int = 0, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Decode attention for sequences sharing their first shared_len tokens (pages
    shared_pages, int32 [shared_len / P]); the shared part is attended once per kv
    head for all sequences, then merged with each sequence's own part."""
    _require(q, "q", torch.bfloat16)
    _require(shared_pages, "shared_pages", torch.int32)
    _require(block_table, "block_table", torch.int32)
    _require(seq_lens, "seq_lens", torch.int32)
    B, Hq = int(q.shape[0]), int(q.shape[1])
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    if out is None:
        out = torch.empty_like(q)
    _require(out, "out", torch.bfloat16)
    if workspace is None:
        n = cascade_workspace_bytes(cache, B, Hq, shared_len, num_splits)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=cache.pool.device)
    _require(workspace, "workspace", torch.uint8)
    rc = _lib.nvfp4_cascade_decode_attention(cache.desc, _ptr(q), B, Hq, _ptr(shared_pages), int(shared_len),
                                             _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
                                             float(sm_scale), _ptr(out), _ptr(workspace), workspace.numel(),
                                             int(num_splits), _stream(stream))
    _check(rc, "nvfp4_cascade_decode_attention")
    return out


def paged_decode_attention_noalloc(cache: PagedCache, q: torch.Tensor, block_table: torch.Tensor,
                                   seq_lens: torch.Tensor, sm_scale: Optional[float] = None,
                                   out: Optional[torch.Tensor] = None, num_splits: int = 0,
                                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Same as paged_decode_attention, with the split scratch taken from the
    library's static device array instead of a workspace, for callers that
    cannot allocate device memory.  `out` must then be provided by the caller
    too (passing None allocates it here, through torch)."""
    _require(q, "q", torch.bfloat16)
    _require(block_table, "block_table", torch.int32)
    _require(seq_lens, "seq_lens", torch.int32)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    if out is None:
        out = torch.empty_like(q)
    _require(out, "out", torch.bfloat16)
    rc = _lib.nvfp4_paged_decode_attention_noalloc(cache.desc, _ptr(q), int(q.shape[0]), int(q.shape[1]),
                                                   _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
                                                   float(sm_scale), _ptr(out), int(num_splits), _stream(stream))
    _check(rc, "nvfp4_paged_decode_attention_noalloc")
    return out


def prefix_dequant(cache: PagedCache, block_table: torch.Tensor, prefix_lens: torch.Tensor,
                   cu_prefix_lens: torch.Tensor, total_prefix_tokens: int, k_ws: Optional[torch.Tensor] = None,
                   v_ws: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """Returns (k_ws, v_ws), BF16 [total][Hkv][128]."""
    _require(block_table, "block_table", torch.int32)
    _require(prefix_lens, "prefix_lens", torch.int32)
    _require(cu_prefix_lens, "cu_prefix_lens", torch.int32)
    shape = (int(total_prefix_tokens), cache.num_kv_heads, HEAD_DIM)
    dev = cache.pool.device
    if k_ws is None:
        k_ws = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    if v_ws is None:
        v_ws = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    _require(k_ws, "k_ws", torch.bfloat16)
    _require(v_ws, "v_ws", torch.bfloat16)
    rc = _lib.nvfp4_prefix_dequant(cache.desc, _ptr(block_table), int(block_table.shape[1]), _ptr(prefix_lens),
                                   _ptr(cu_prefix_lens), int(prefix_lens.shape[0]), int(total_prefix_tokens),
                                   _ptr(k_ws), _ptr(v_ws), _stream(stream))
    _check(rc, "nvfp4_prefix_dequant")
    return k_ws, v_ws


def profile_decode(before, after, every: int = 1):
    """Benchmark hook: record torch.cuda.Event pairs around the decode-kernel
    launch of every `every`-th following call (the j-th such call uses pair
    j % len).  Pass empty lists to stop."""
    if not before:
        _check(_lib.nvfp4kv_profile_decode(None, None, 0, 1), "nvfp4kv_profile_decode")
        return
    n = len(before)
    assert len(after) == n
    for e in list(before) + list(after):
        if not e.cuda_event:      # torch creates the CUDA event on first record
            e.record()
    arr_b = (ctypes.c_void_p * n)(*[e.cuda_event for e in before])
    arr_a = (ctypes.c_void_p * n)(*[e.cuda_event for e in after])
    _check(_lib.nvfp4kv_profile_decode(arr_b, arr_a, n, int(every)), "nvfp4kv_profile_decode")


def selftest_bounded_wait(arrive: bool, poll_limit: int, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Failure-path self-test: one warp waits (at most poll_limit polls) on an
    mbarrier phase that completes only if `arrive`.  Returns a device int32
    tensor [1]: 1 if the wait gave up (the device error word then holds the
    timeout bit), else 0."""
    result = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _check(_lib.nvfp4kv_selftest_bounded_wait(1 if arrive else 0, int(poll_limit), _ptr(result), _stream(stream)),
           "nvfp4kv_selftest_bounded_wait")
    return result


def extend_attention(q: torch.Tensor, k_prefix: torch.Tensor, v_prefix: torch.Tensor, cu_prefix_lens: torch.Tensor,
                     k_chunk: torch.Tensor, v_chunk: torch.Tensor, cu_q_lens: torch.Tensor, max_q_len: int,
                     sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Each request's chunk attends to [its prefix rows || the chunk], causally in
    the chunk.  q: BF16 [total_q][Hq][128]; k_prefix, v_prefix: BF16
    [total_prefix][Hkv][128] (e.g. from prefix_dequant); k_chunk, v_chunk: BF16
    [total_q][Hkv][128]; cu_*: int32 [R+1]; max_q_len: bound on chunk lengths."""
    for name, x in (("q", q), ("k_prefix", k_prefix), ("v_prefix", v_prefix), ("k_chunk", k_chunk),
                    ("v_chunk", v_chunk)):
        if not x.is_cuda or x.dtype != torch.bfloat16 or not x.is_contiguous() or x.dim() != 3 or x.shape[2] != HEAD_DIM:
            raise ValueError("%s must be a contiguous CUDA bfloat16 tensor [rows][heads][128]" % name)
    _require(cu_prefix_lens, "cu_prefix_lens", torch.int32)
    _require(cu_q_lens, "cu_q_lens", torch.int32)
    R = int(cu_q_lens.shape[0]) - 1
    if int(cu_prefix_lens.shape[0]) != R + 1:
        raise ValueError("cu_prefix_lens and cu_q_lens must have the same length")
    hq, hkv = int(q.shape[1]), int(k_chunk.shape[1])
    if k_prefix.shape[1] != hkv or v_prefix.shape[1] != hkv or v_chunk.shape[1] != hkv:
        raise ValueError("K/V head counts differ")
    if k_chunk.shape[0] != q.shape[0] or v_chunk.shape[0] != q.shape[0]:
        raise ValueError("chunk K/V must have one row per query token")
    if out is None:
        out = torch.empty_like(q)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    # an empty prefix still needs a valid aligned pointer
    kp = k_prefix if k_prefix.numel() else torch.zeros((1, hkv, HEAD_DIM), dtype=torch.bfloat16, device=q.device)
    vp = v_prefix if v_prefix.numel() else kp
    rc = _lib.nvfp4_extend_attention(_ptr(q), _ptr(kp), _ptr(vp), _ptr(cu_prefix_lens), int(kp.shape[0]),
                                     _ptr(k_chunk), _ptr(v_chunk), _ptr(cu_q_lens), int(q.shape[0]), R,
                                     int(max_q_len), hq, hkv, float(sm_scale), _ptr(out), _stream(stream))
    _check(rc, "nvfp4_extend_attention")
    return out


def extend_attention_paged(cache: PagedCache, q: torch.Tensor, block_table: torch.Tensor, prefix_lens: torch.Tensor,
                           k_chunk: torch.Tensor, v_chunk: torch.Tensor, cu_q_lens: torch.Tensor, max_q_len: int,
                           sm_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                           stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """extend_attention with request r's prefix read from the NVFP4 cache: tokens
    0 .. prefix_lens[r] - 1 of its pages (block_table row r, int32 [R][max_pages]),
    expanded to BF16 inside the kernel; equals prefix_dequant + extend_attention."""
    for name, x in (("q", q), ("k_chunk", k_chunk), ("v_chunk", v_chunk)):
        if not x.is_cuda or x.dtype != torch.bfloat16 or not x.is_contiguous() or x.dim() != 3 or x.shape[2] != HEAD_DIM:
            raise ValueError("%s must be a contiguous CUDA bfloat16 tensor [rows][heads][128]" % name)
    _require(block_table, "block_table", torch.int32)
    _require(prefix_lens, "prefix_lens", torch.int32)
    _require(cu_q_lens, "cu_q_lens", torch.int32)
    R = int(cu_q_lens.shape[0]) - 1
    if int(prefix_lens.shape[0]) != R or int(block_table.shape[0]) != R:
        raise ValueError("prefix_lens and block_table need one entry / row per request")
    hq = int(q.shape[1])
    if k_chunk.shape[1] != cache.num_kv_heads or v_chunk.shape[1] != cache.num_kv_heads:
        raise ValueError("chunk K/V must have the cache's kv heads")
    if k_chunk.shape[0] != q.shape[0] or v_chunk.shape[0] != q.shape[0]:
        raise ValueError("chunk K/V must have one row per query token")
    if out is None:
        out = torch.empty_like(q)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(HEAD_DIM)
    rc = _lib.nvfp4_extend_attention_paged(cache.desc, _ptr(q), _ptr(block_table), int(block_table.shape[1]),
                                           _ptr(prefix_lens), _ptr(k_chunk), _ptr(v_chunk), _ptr(cu_q_lens),
                                           int(q.shape[0]), R, int(max_q_len), hq, float(sm_scale), _ptr(out),
                                           _stream(stream))
    _check(rc, "nvfp4_extend_attention_paged")
    return out


def check_device_errors(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise the stream and return (and clear) the device error status (0 = none)."""
    return int(_lib.nvfp4kv_check_device_errors(_stream(stream)))
