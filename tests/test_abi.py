"""The C-ABI library builds for sm_103a, loads, exports every function that
include/w4a16.h declares, and rejects bad arguments on the host before any
CUDA call (these checks need no GPU: validation runs first)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")

nvcc_missing = shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc")


@pytest.fixture(scope="module")
def lib():
    if nvcc_missing:
        pytest.skip("nvcc not available")
    from int4_weight_only_gemm_gb300 import _build
    path = _build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(w4a16_[a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("w4a16_pack", "w4a16_unpack", "w4a16_gemm", "w4a16_workspace_bytes",
                 "w4a16_set_workspace", "w4a16_status_str", "w4a16_last_device_status"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in w4a16.h but not exported"


def test_status_strings(lib):
    lib.w4a16_status_str.restype = ctypes.c_char_p
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = lib.w4a16_status_str(code).decode()
        assert s and s != "unknown status"
    assert lib.w4a16_status_str(42).decode() == "unknown status"


def _gemm(lib, x, q, s, z, M, N, K, g, y):
    vp = ctypes.c_void_p
    lib.w4a16_gemm_ws.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  vp, vp, ctypes.c_size_t, vp]
    return lib.w4a16_gemm_ws(x, q, s, z, M, N, K, g, y, None, 0, None)


A, B, C, D, E = 0x10000, 0x200000, 0x3000000, 0x40000000, 0x500000000  # distinct aligned fake addresses


def test_host_validation_rejects_before_launch(lib):
    # null pointers
    assert _gemm(lib, None, B, C, D, 1, 128, 256, 128, E) == -1
    assert _gemm(lib, A, B, C, D, 1, 128, 256, 128, None) == -1
    # bad sizes
    assert _gemm(lib, A, B, C, D, -1, 128, 256, 128, E) == -1
    assert _gemm(lib, A, B, C, D, 1, 12, 256, 128, E) == -1       # N % 8
    assert _gemm(lib, A, B, C, D, 1, 0, 256, 128, E) == -1
    # unsupported group / K
    assert _gemm(lib, A, B, C, D, 1, 128, 256, 64, E) == -3
    assert _gemm(lib, A, B, C, D, 1, 128, 320, 128, E) == -3
    # alignment
    assert _gemm(lib, A + 2, B, C, D, 1, 128, 256, 128, E) == -2
    assert _gemm(lib, A, B + 4, C, D, 1, 128, 256, 128, E) == -2
    assert _gemm(lib, A, B, C, D, 1, 128, 256, 128, E + 8) == -2
    # output overlapping an input
    assert _gemm(lib, A, B, C, D, 1, 128, 256, 128, A + 256) == -1


def test_empty_batch_is_a_checked_no_op(lib):
    """M == 0 computes nothing: the shape is still checked, no pointer is read
    (null pointers pass), and the call returns before any CUDA call -- which
    is why it succeeds here, without a GPU."""
    assert _gemm(lib, None, None, None, None, 0, 128, 256, 128, None) == 0
    assert _gemm(lib, None, None, None, None, 0, 12, 256, 128, None) == -1   # N % 8
    assert _gemm(lib, None, None, None, None, 0, 128, 320, 128, None) == -3  # K % 128
    assert _gemm(lib, None, None, None, None, 0, 128, 256, 64, None) == -3   # group
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.w4a16_gemm_ex.argtypes = [i, ctypes.c_uint, vp, vp, vp, vp, i, i, i, i, vp, vp, ctypes.c_size_t, vp]
    assert lib.w4a16_gemm_ex(0, 0, None, None, None, None, 0, 128, 256, 128, None, None, 0, None) == 0
    assert lib.w4a16_gemm_ex(9, 0, None, None, None, None, 0, 128, 256, 128, None, None, 0, None) == -1  # path
    assert lib.w4a16_gemm_ex(0, 1 << 30, None, None, None, None, 0, 128, 256, 128, None, None, 0, None) == -1  # flags
    lib.w4a16_gemm_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, vp, vp]
    assert lib.w4a16_gemm_noalloc(None, None, None, None, 0, 128, 256, 128, None, None) == 0
    lib.w4a16_gemm_gate_up_silu.argtypes = [i, ctypes.c_uint, vp, vp, vp, vp, i, i, i, i, vp, vp, ctypes.c_size_t, vp]
    assert lib.w4a16_gemm_gate_up_silu(0, 0, None, None, None, None, 0, 64, 256, 128, None, None, 0, None) == 0
    lib.w4a16_workspace_bytes.restype = ctypes.c_size_t
    lib.w4a16_workspace_bytes.argtypes = [i, i, i, i]
    assert lib.w4a16_workspace_bytes(0, 128, 256, 128) == 0


def test_pack_validation(lib):
    vp = ctypes.c_void_p
    lib.w4a16_pack.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, vp]
    lib.w4a16_unpack.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, vp]
    assert lib.w4a16_pack(None, B, 256, 128, None) == -1
    assert lib.w4a16_pack(A, B, 256, 12, None) == -1
    assert lib.w4a16_pack(A, B, 200, 128, None) == -3
    assert lib.w4a16_pack(A + 4, B, 256, 128, None) == -2
    assert lib.w4a16_pack(A, A + 16, 256, 128, None) == -1     # overlap
    assert lib.w4a16_unpack(A, None, 256, 128, None) == -1


def test_binding_imports_without_gpu(lib):
    import int4_weight_only_gemm_gb300 as w
    assert w.load_library() is not None
    assert w.w4a16_status_str(-5).startswith("a bounded")


def test_gate_up_validation(lib):
    vp, ci, cu, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
    lib.w4a16_pack_gate_up.argtypes = [vp, vp, ci, ci, vp]
    lib.w4a16_unpack_gate_up.argtypes = [vp, vp, ci, ci, vp]
    lib.w4a16_gemm_gate_up_silu.argtypes = [ci, cu, vp, vp, vp, vp, ci, ci, ci, ci, vp, vp, sz, vp]
    assert lib.w4a16_pack_gate_up(None, B, 256, 64, None) == -1
    assert lib.w4a16_pack_gate_up(A, B, 256, 0, None) == -1
    assert lib.w4a16_pack_gate_up(A, B, 256, 32, None) == -3      # H % 64
    assert lib.w4a16_pack_gate_up(A, B, 200, 64, None) == -3      # K % 128
    assert lib.w4a16_pack_gate_up(A + 4, B, 256, 64, None) == -2
    assert lib.w4a16_pack_gate_up(A, A + 16, 256, 64, None) == -1  # overlap
    assert lib.w4a16_unpack_gate_up(A, None, 256, 64, None) == -1

    def gu(x, y, M=1, H=64, K=256, group=128, flags=1):
        return lib.w4a16_gemm_gate_up_silu(0, flags, x, B, C, D, M, H, K, group, y, None, 0, None)

    assert gu(None, E) == -1
    assert gu(A, None) == -1
    assert gu(A, E, H=0) == -1
    assert gu(A, E, H=96) == -3       # H % 64
    assert gu(A, E, K=320) == -3      # K % 128
    assert gu(A, E, group=64) == -3
    assert gu(A, E, flags=4) == -1    # unknown flag bit
    assert gu(A + 2, E) == -2
    assert gu(A, E + 8) == -2
    assert gu(A, A + 64) == -1        # y [1][64] bf16 overlapping x


def test_requant_validation(lib):
    vp, ci = ctypes.c_void_p, ctypes.c_int
    lib.w4a16_requant_pack.argtypes = [vp, vp, vp, ci, ci, ci, vp, vp]
    assert lib.w4a16_requant_pack(None, C, D, 256, 128, 128, B, None) == -1
    assert lib.w4a16_requant_pack(A, C, D, 256, 128, 64, B, None) == -3
    assert lib.w4a16_requant_pack(A, C, D, 256, 12, 128, B, None) == -1
    assert lib.w4a16_requant_pack(A + 2, C, D, 256, 128, 128, B, None) == -2
    assert lib.w4a16_requant_pack(A, C, D, 256, 128, 128, A + 16, None) == -1  # codes over w
