"""Failure detection without a GPU fault: a bounded device-side wait on a
barrier that nothing completes must end with W4A16_ETIMEOUT reported to the
host, and the context must stay usable for the next GEMM."""
import pytest
import torch

import w4a16_inputs as wi
from tests.gpu_helpers import Device, bf16_to_f64, check_close

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import int4_weight_only_gemm_gb300 as w
    lib = w.load_library()
    import ctypes
    lib.w4a16_selftest_wait_timeout.argtypes = [ctypes.c_longlong, ctypes.c_void_p]
    assert w.w4a16_last_device_status() == 0
    st = lib.w4a16_selftest_wait_timeout(20_000_000, torch.cuda.current_stream().cuda_stream)  # 20 ms
    assert st == 0
    assert w.w4a16_last_device_status() == w.W4A16_ETIMEOUT
    assert w.w4a16_last_device_status() == 0  # read clears it
    # the context is still usable
    import oracle
    p = wi.generate_named("tiny", 1, 0)
    y = Device(p).run()
    check_close(bf16_to_f64(y), oracle.gemm(p.x, p.qweight, p.scales, p.qzeros), "after timeout")


def test_selftest_rejects_bad_limit():
    import ctypes
    import int4_weight_only_gemm_gb300 as w
    lib = w.load_library()
    lib.w4a16_selftest_wait_timeout.argtypes = [ctypes.c_longlong, ctypes.c_void_p]
    assert lib.w4a16_selftest_wait_timeout(10, None) == w.W4A16_EINVAL
    assert lib.w4a16_selftest_wait_timeout(10 ** 12, None) == w.W4A16_EINVAL
