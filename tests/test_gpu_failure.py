"""Failure detection on the GPU without a fault: a bounded wait on an mbarrier
phase that nothing completes gives up after its poll limit, reports the timeout
through the device error word and returns, and the context stays usable (a
decode afterwards still matches the oracle)."""

import pytest
import torch

import workloads
from gpu_common import check_attention, decode_both, fill_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import nvfp4_quantised_paged_gb300 as mod
    return mod


def test_wait_that_nothing_completes_times_out_and_reports(m):
    assert m.check_device_errors() == 0
    r = m.selftest_bounded_wait(False, 4096)
    torch.cuda.synchronize()
    assert int(r.item()) == 1
    assert m.check_device_errors() == -4      # NVFP4KV_EDEVICE_CHECK: the timeout bit is set
    assert m.check_device_errors() == 0       # and was cleared by the read


def test_wait_that_completes_reports_nothing(m):
    r = m.selftest_bounded_wait(True, 4096)
    torch.cuda.synchronize()
    assert int(r.item()) == 0
    assert m.check_device_errors() == 0


def test_context_usable_after_a_timeout(m):
    r = m.selftest_bounded_wait(False, 64)
    torch.cuda.synchronize()
    assert int(r.item()) == 1 and m.check_device_errors() == -4
    w = workloads.tiny_decode()
    cache, pool = fill_both(w, m)
    out, ref, spread = decode_both(w, m, cache, pool)
    check_attention(out, ref, "decode after a timeout", spread=spread)


def test_selftest_rejects_bad_arguments(m):
    lib = m.library()
    res = torch.zeros(1, dtype=torch.int32, device="cuda")
    import ctypes
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.nvfp4kv_selftest_bounded_wait(0, 0, ctypes.c_void_p(res.data_ptr()), s) == -1
    assert lib.nvfp4kv_selftest_bounded_wait(0, (1 << 24) + 1, ctypes.c_void_p(res.data_ptr()), s) == -1
    assert lib.nvfp4kv_selftest_bounded_wait(0, 16, None, s) == -1
