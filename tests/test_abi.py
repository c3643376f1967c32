"""CPU checks of the C ABI: the library builds, loads, exports every symbol the
header declares, reports the documented layout sizes, and rejects invalid
arguments on the host (no GPU needed: rejected calls launch nothing)."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4kv.h")


def _lib_path():
    import __graft_entry__
    return __graft_entry__._cuda_build_module().build()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^NVFP4KV_API\s+[\w\s\*]*?\b(nvfp4\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_three_paths():
    names = declared_functions()
    for n in ("nvfp4_kv_quantize_append", "nvfp4_paged_decode_attention", "nvfp4_prefix_dequant"):
        assert n in names
    assert len(names) == len(set(names)) >= 10


def test_library_exports_every_declared_symbol():
    path = _lib_path()
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for n in declared_functions():
        assert n in exported, n
    # nothing else leaks out of the library
    assert exported == set(declared_functions())
    lib = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(lib, n)


@pytest.fixture(scope="module")
def m():
    _lib_path()
    import nvfp4_quantised_paged_gb300 as mod
    return mod


def test_binding_exports_match_header(m):
    assert set(m.EXPORTED_SYMBOLS) == set(declared_functions())


def test_slab_sizes_and_byte_ratio(m):
    for P in (16, 32, 64, 128):
        nv, f8 = m.slab_bytes(m.DTYPE_NVFP4, P), m.slab_bytes(m.DTYPE_FP8_E4M3, P)
        assert nv == 144 * P and f8 == 256 * P and nv / f8 == 0.5625
    for bad in (8, 48, 256):
        with pytest.raises(m.NVFP4KVError):
            m.slab_bytes(m.DTYPE_NVFP4, bad)


def _desc(m, **kw):
    d = dict(pool=4096, num_pages=4, page_size=16, num_kv_heads=2, head_dim=128, dtype=0, k_global_scale=1.0,
             v_global_scale=1.0)
    d.update(kw)
    return m._CacheDesc(d["pool"], d["num_pages"], d["page_size"], d["num_kv_heads"], d["head_dim"], d["dtype"],
                        d["k_global_scale"], d["v_global_scale"])


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), -2), (dict(page_size=48), -2), (dict(dtype=7), -2), (dict(num_kv_heads=0), -1),
    (dict(k_global_scale=0.0), -1), (dict(v_global_scale=float("inf")), -1), (dict(pool=4097), -1),
    (dict(k_global_scale=1e-40), -1), (dict(v_global_scale=-2.0), -1), (dict(k_global_scale=float("nan")), -1),
    (dict(pool=0), -1), (dict(num_pages=0), -1),
])
def test_invalid_cache_descriptors_are_rejected_before_any_launch(m, kw, status):
    lib = m.library()
    d = _desc(m, **kw)
    P = ctypes.c_void_p
    rc = lib.nvfp4_kv_quantize_append(ctypes.byref(d), P(4096), P(4096), 1, 256, P(4096), None)
    assert rc == status
    rc = lib.nvfp4_paged_decode_attention(ctypes.byref(d), P(4096), 1, 2, P(4096), 1, P(4096), 0.1, P(4096),
                                          P(4096), 1 << 20, 0, None)
    assert rc == status
    rc = lib.nvfp4_prefix_dequant(ctypes.byref(d), P(4096), 1, P(4096), P(4096), 1, 16, P(4096), P(4096), None)
    assert rc == status


def test_invalid_call_arguments_are_rejected(m):
    lib = m.library()
    d = ctypes.byref(_desc(m))
    P = ctypes.c_void_p
    # append: stride too small, stride not a multiple of 8, misaligned k, null slot mapping, negative count
    assert lib.nvfp4_kv_quantize_append(d, P(4096), P(4096), 1, 128, P(4096), None) == -1
    assert lib.nvfp4_kv_quantize_append(d, P(4096), P(4096), 1, 260, P(4096), None) == -1
    assert lib.nvfp4_kv_quantize_append(d, P(4098), P(4096), 1, 256, P(4096), None) == -1
    assert lib.nvfp4_kv_quantize_append(d, P(4096), P(4096), 1, 256, None, None) == -1
    assert lib.nvfp4_kv_quantize_append(d, P(4096), P(4096), -1, 256, P(4096), None) == -1
    assert lib.nvfp4_kv_quantize_append(d, None, None, 0, 256, None, None) == 0  # empty call is a no-op
    # decode: heads not a multiple of kv heads, group > 16, misaligned workspace, bad sm_scale, empty batch
    assert lib.nvfp4_paged_decode_attention(d, P(4096), 1, 3, P(4096), 1, P(4096), 0.1, P(4096), P(4096), 1 << 20,
                                            0, None) == -1
    assert lib.nvfp4_paged_decode_attention(d, P(4096), 1, 34, P(4096), 1, P(4096), 0.1, P(4096), P(4096), 1 << 20,
                                            0, None) == -2
    assert lib.nvfp4_paged_decode_attention(d, P(4096), 1, 2, P(4096), 1, P(4096), 0.1, P(4096), P(4100), 1 << 20,
                                            1, None) == -1
    assert lib.nvfp4_paged_decode_attention(d, P(4096), 1, 2, P(4096), 1, P(4096), float("nan"), P(4096),
                                            P(4096), 1 << 20, 1, None) == -1
    assert lib.nvfp4_paged_decode_attention(d, None, 0, 2, None, 1, None, 0.1, None, None, 0, 0, None) == 0
    # prefix dequant: misaligned workspace, negative total, nothing to do
    assert lib.nvfp4_prefix_dequant(d, P(4096), 1, P(4096), P(4096), 1, 16, P(4098), P(4096), None) == -1
    assert lib.nvfp4_prefix_dequant(d, P(4096), 1, P(4096), P(4096), 1, -1, P(4096), P(4096), None) == -1
    assert lib.nvfp4_prefix_dequant(d, None, 1, None, None, 0, 0, None, None, None) == 0


def test_status_strings(m):
    lib = m.library()
    for s in (0, -1, -2, -3, -4):
        assert lib.nvfp4kv_status_string(s)
    assert lib.nvfp4kv_version() >= 100


def test_paged_extend_and_launch_count_arguments(m):
    lib = m.library()
    d = ctypes.byref(_desc(m))
    f8 = ctypes.byref(_desc(m, dtype=1))
    P = ctypes.c_void_p
    # paged extend: (cache, q, block_table, max_pages, prefix_lens, k_chunk, v_chunk, cu_q, total_q, num_reqs,
    # max_q_len, num_q_heads, sm_scale, out, stream)
    args = [P(4096), P(4096), 4, P(4096), P(4096), P(4096), P(4096), 16, 1, 16, 8, 0.1, P(4096), None]
    ok_args = list(args)
    assert lib.nvfp4_extend_attention_paged(f8, *ok_args) == -2  # an NVFP4 pool only
    bad = list(args); bad[10] = 3                                # heads not a multiple of kv heads
    assert lib.nvfp4_extend_attention_paged(d, *bad) == -1
    bad = list(args); bad[2] = 0                                 # no pages per request
    assert lib.nvfp4_extend_attention_paged(d, *bad) == -1
    bad = list(args); bad[0] = P(4098)                           # misaligned q
    assert lib.nvfp4_extend_attention_paged(d, *bad) == -1
    bad = list(args); bad[11] = float("nan")
    assert lib.nvfp4_extend_attention_paged(d, *bad) == -1
    bad = list(args); bad[8] = 0                                 # no requests: nothing to do
    assert lib.nvfp4_extend_attention_paged(d, *bad) == 0
    # launch count: decode + reduction for a batch of up to 96 (planned in the decode CTAs), the plan
    # kernel as well for a larger one, and the shared-prefix kernel for a cascade call (planned by the plan kernel)
    assert lib.nvfp4kv_decode_launch_count(d, 4, 8, 0, 0) == 2
    assert lib.nvfp4kv_decode_launch_count(d, 96, 8, 0, 0) == 2
    assert lib.nvfp4kv_decode_launch_count(d, 97, 8, 0, 0) == 3
    assert lib.nvfp4kv_decode_launch_count(d, 4, 8, 0, 128) == 4
    assert lib.nvfp4kv_decode_launch_count(d, 0, 8, 0, 0) == 0
    assert lib.nvfp4kv_decode_launch_count(d, 4, 3, 0, 0) == 0


def test_binding_refuses_host_tensors(m):
    """The product path has no CPU fallback: host tensors are rejected before
    any library call, for the pool and for every per-call input."""
    import torch
    with pytest.raises(ValueError):
        m.PagedCache(4, 16, 1, device="cpu")
    pool = torch.zeros((4, 1, m.slab_bytes(m.DTYPE_NVFP4, 16)), dtype=torch.uint8)
    with pytest.raises(ValueError):
        m.PagedCache(4, 16, 1, pool=pool)
    k = torch.zeros((2, 1, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        m.calibrate_global_scales(k, k, 1)


def test_header_is_plain_c(tmp_path):
    """The boundary is a C ABI: the header compiles as C11 (no C++ or torch
    types), and every declared entry point links against the library from C."""
    import shutil
    cuda_inc = "/usr/local/cuda/include"
    if not shutil.which("gcc") or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA headers are missing")
    names = declared_functions()
    src = tmp_path / "use_header.c"
    src.write_text('#include "nvfp4kv.h"\ntypedef void (*fn_t)(void);\nstatic const fn_t fns[] = {\n' +
                   "".join("    (fn_t)&%s,\n" % n for n in names) +
                   "};\nint main(void) {\n    int ok = 1;\n    for (unsigned i = 0; i < sizeof fns / sizeof fns[0]; i++)"
                   " ok &= fns[i] != 0;\n    return ok ? 0 : 1;\n}\n")
    lib = _lib_path()
    exe = tmp_path / "use_header"
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                        "-I", cuda_inc, str(src), "-o", str(exe), "-L", os.path.dirname(lib), "-lnvfp4kv",
                        "-Wl,-rpath," + os.path.dirname(lib)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert subprocess.run([str(exe)]).returncode == 0


def _declared_signatures():
    """{name: (return C type, [parameter C types])} parsed from the header."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    sigs = {}
    for ret, name, params in re.findall(r"NVFP4KV_API\s+([\w\s\*]+?)\s*\b(nvfp4\w+)\s*\(([^)]*)\)\s*;", text):
        params = " ".join(params.split())
        types = [] if params in ("", "void") else [re.sub(r"\s*\b\w+$", "", p.strip()) for p in params.split(",")]
        sigs[name] = (ret.strip(), types)
    return sigs


def _ctype_of(c):
    """The ctypes class a C parameter type must be declared with."""
    if c.replace(" ", "") == "constnvfp4kv_cache*":
        return "desc"
    if "*" in c or c in ("cudaStream_t",):
        return ctypes.c_void_p
    return {"int": ctypes.c_int, "unsigned": ctypes.c_uint, "int64_t": ctypes.c_int64, "size_t": ctypes.c_size_t,
            "float": ctypes.c_float}[c]


def test_binding_argtypes_match_the_header(m):
    """Every ctypes signature of the binding has the header's parameter count
    and types (a mismatch would shift arguments silently)."""
    lib = m.library()
    sigs = _declared_signatures()
    assert set(sigs) == set(declared_functions())
    for name, (ret, params) in sigs.items():
        fn = getattr(lib, name)
        assert len(fn.argtypes) == len(params), name
        for got, c in zip(fn.argtypes, params):
            want = _ctype_of(c)
            if want == "desc":
                assert got is ctypes.POINTER(m._CacheDesc), (name, c)
            else:
                assert got is want, (name, c, got)
        want_ret = {"int": ctypes.c_int, "size_t": ctypes.c_size_t, "const char *": ctypes.c_char_p}[ret]
        assert fn.restype is want_ret, (name, ret)


def test_noalloc_scratch_size_matches_the_header(m):
    text = open(HEADER).read()
    mo = re.search(r"#define\s+NVFP4KV_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert mo and m.NOALLOC_SCRATCH_BYTES == int(mo.group(1)) << int(mo.group(2))
