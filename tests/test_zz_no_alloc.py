"""The no-allocation entry point, w4a16_gemm_noalloc, against the oracle and the regular one.

w4a16_gemm_noalloc is for callers that may not allocate device memory (for
example a plugin inside a runtime that plans all device memory itself): it
runs the split-K GEMV with the scratch array compiled into the library
instead of a caller-provided workspace.  This file runs last (pytest collects
it after the others) and must pass both alone and after the rest.
"""
import ctypes
import os
import re

import pytest
import torch

import oracle
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
def test_noalloc_matches_oracle_and_regular_entry_point_twice(shape, M):
    """Two calls in a row (sharing, and reusing, the built-in scratch) match
    the oracle within the GEMM tolerance and the regular entry point (caller
    workspace, same kernel) bit for bit; each counts one launch."""
    w, lib = _lib()
    p = wi.generate_named(shape, M, 50)
    d = Device(p)
    ref = oracle.gemm(p.x, p.qweight, p.scales, p.qzeros)
    regular = d.run(w.PATH_GEMV_SPLITK)  # the same split-K kernel with a caller workspace
    for call in range(2):
        y = torch.full((M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        n0 = w.w4a16_launch_count()
        assert _noalloc(lib, d, M, y) == 0
        assert w.w4a16_launch_count() == n0 + 1
        torch.cuda.synchronize()
        check_close(bf16_to_f64(y), ref, f"noalloc {shape} M={M} call {call}")
        assert torch.equal(y.view(torch.int16), regular.view(torch.int16))
    assert w.w4a16_last_device_status() == 0


def test_noalloc_allocates_no_device_memory():
    """After a first call (which looks up the array's address), further calls
    leave the device's free memory unchanged."""
    w, lib = _lib()
    p = wi.generate_named("o_proj", 2, 52)
    d = Device(p)
    y = torch.empty((2, p.N), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, d, 2, y) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        assert _noalloc(lib, d, 2, y) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_noalloc_scratch_covers_every_gemv_problem():
    """The built-in array holds the split-K scratch of every M <= 8 problem of
    the decoder's shapes, the vocabulary head included."""
    w, _ = _lib()
    limit = _scratch_limit()
    for shape in list(wi.LAYER) + ["vocab"]:
        K, N = wi.shape_kn(shape)
        for M in range(1, 9):
            assert w.w4a16_workspace_bytes(M, N, K, path=w.PATH_GEMV_SPLITK) <= limit, (shape, M)


def test_noalloc_rejects_what_it_cannot_run():
    w, lib = _lib()
    p = wi.generate_named("qkv", 9, 51)
    d = Device(p)
    y = torch.empty((9, p.N), dtype=torch.bfloat16, device="cuda")
    n0 = w.w4a16_launch_count()
    assert _noalloc(lib, d, 9, y) == w.W4A16_EUNSUPPORTED  # beyond the GEMV's M
    assert lib.w4a16_gemm_noalloc(None, None, None, None, 1, 128, 256, 128, None, None) == w.W4A16_EINVAL
    assert _noalloc(lib, d, -1, y) == w.W4A16_EINVAL
    assert _noalloc(lib, d, 0, y) == w.W4A16_OK  # an empty batch: nothing to compute
    assert w.w4a16_launch_count() == n0
