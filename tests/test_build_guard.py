"""Build-time guard on the decode kernel's register allocation.

The NVFP4 decode kernel (group <= 8) runs at its 128-register cap so that
eight CTAs fit on an SM.  At that cap ptxas spills a few bytes outside the
main loop; an edit anywhere in the kernel (its prologue included) can change
the allocation so that values used inside the loop are reloaded from local
memory on every chunk, which made the 32K decode about 1.5x slower in one
such build (586 against 379 us) while every numerical test still passed.  This
compiles the kernel as the library build does and bounds its spills."""

import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "nvfp4_quantised_paged_gb300", "csrc")
MAX_SPILL_BYTES = 4


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else shutil.which("nvcc")


def test_decode_kernel_spills_stay_small(tmp_path):
    nvcc = _nvcc()
    if not nvcc:
        pytest.skip("nvcc not available")
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo",
                        "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-Xptxas", "-v", "-c",
                        os.path.join(CSRC, "decode_attention.cu"), "-o", str(tmp_path / "d.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = r.stderr.splitlines()
    found = 0
    for i, line in enumerate(lines):
        # decode_kernel<NVFP4 (0), one N tile (1)>: the kernel of every workload with G <= 8
        if "Function properties for" in line and "decode_kernelILi0ELi1E" in line:
            m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", lines[i + 1])
            assert m, lines[i + 1]
            stores, loads = int(m.group(1)), int(m.group(2))
            assert stores <= MAX_SPILL_BYTES and loads <= MAX_SPILL_BYTES, (stores, loads)
            found += 1
    assert found == 1
