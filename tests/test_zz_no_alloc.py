"""The no-allocation entry point, w4a16_gemm_noalloc, against the regular one.

w4a16_gemm_noalloc is for callers that may not allocate device memory (for
example a plugin inside a runtime that plans all device memory itself): it
runs the split-K GEMV with the scratch array compiled into the library
instead of a caller-provided workspace.  This file runs last (pytest collects
it after the others) and must pass both alone and after the rest.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import w4a16_inputs as wi
from tests.gpu_helpers import Device, bf16_to_f64, check_close

pytestmark = pytest.mark.gpu

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "w4a16.h")


def _scratch_limit():
    m = re.search(r"#define\s+W4A16_NOALLOC_SCRATCH_BYTES\s+\(?(\d+)u?\s*<<\s*(\d+)\)?", open(HEADER).read())
    return int(m.group(1)) << int(m.group(2))


def _lib():
    import int4_weight_only_gemm_gb300 as w
    lib = w.load_library()
    vp, ci = ctypes.c_void_p, ctypes.c_int
    lib.w4a16_gemm_noalloc.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, vp, vp]
    return w, lib


def _noalloc(lib, d, M, y):
    p = d.prob
    return lib.w4a16_gemm_noalloc(d.x.data_ptr(), d.qd.data_ptr(), d.scales.data_ptr(), d.qzeros.data_ptr(),
                                  M, p.N, p.K, 128, y.data_ptr(), torch.cuda.current_stream().cuda_stream)


CASES = [("qkv", 1), ("down", 2), ("gate_up", 4), ("o_proj", 3)]


@pytest.mark.parametrize("shape,M", CASES)
def test_noalloc_matches_regular_entry_point_twice(shape, M):
    w, lib = _lib()
    p = wi.generate_named(shape, M, 50)
    d = Device(p)
    need = w.w4a16_workspace_bytes(M, p.N, p.K, path=w.PATH_GEMV)
    if need > _scratch_limit():
        pytest.skip("this problem needs more scratch than the built-in array holds")
    want = bf16_to_f64(d.run(w.PATH_GEMV))  # the regular entry point, caller workspace
    for call in range(2):  # two calls in a row share (and reuse) the built-in scratch
        y = torch.full((M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(lib, d, M, y) == 0
        torch.cuda.synchronize()
        check_close(bf16_to_f64(y), want, f"noalloc {shape} M={M} call {call}")
    assert w.w4a16_last_device_status() == 0


def test_noalloc_rejects_what_it_cannot_run():
    w, lib = _lib()
    p = wi.generate_named("qkv", 9, 51)
    d = Device(p)
    y = torch.empty((9, p.N), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, d, 9, y) == w.W4A16_EUNSUPPORTED  # beyond the GEMV's M
    # a problem whose split-K scratch exceeds the array is refused, not run
    limit = _scratch_limit()
    for M in (8, 4, 2):
        need = w.w4a16_workspace_bytes(M, p.N, p.K, path=w.PATH_GEMV)
        if need > limit:
            y = torch.empty((M, p.N), dtype=torch.bfloat16, device="cuda")
            assert _noalloc(lib, d, M, y) == w.W4A16_EWORKSPACE
            break
    assert lib.w4a16_gemm_noalloc(None, None, None, None, 1, 128, 256, 128, None, None) == w.W4A16_EINVAL
