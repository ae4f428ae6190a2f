"""Python binding of the W4A16 group-quantized GEMM library (libw4a16.so).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/w4a16.h.  PyTorch supplies device
memory and streams.  There is no fallback: if the compiled library is missing
or a call fails, an exception is raised.

    y[m][n] = sum_k x[m][k] * (q[k][n] - z[k/128][n]) * s[k/128][n]

Tensors (all on one CUDA device, contiguous):
    x        [M, K]    torch.bfloat16
    qweight  [K/8, N]  torch.int32   canonical packing (bits 4i..4i+3 = row 8j+i)
    qweight_dev        torch.int32   device layout from w4a16_pack (same size)
    scales   [K/128, N] torch.float16
    qzeros   [K/128, N/8] torch.int32 (bits 4i..4i+3 = column 8c+i)
    y        [M, N]    torch.bfloat16
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw4a16.so")

W4A16_OK = 0
W4A16_EINVAL = -1
W4A16_EALIGN = -2
W4A16_EUNSUPPORTED = -3
W4A16_ECUDA = -4
W4A16_ETIMEOUT = -5
W4A16_EWORKSPACE = -6
PATH_AUTO, PATH_GEMV, PATH_TC, PATH_GEMV_SPLITK, PATH_GEMV_CS = 0, 1, 2, 3, 4
FLAG_PDL, FLAG_STATIC_WEIGHTS = 1, 2

_lib = None
_lock = threading.Lock()


class W4A16Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {w4a16_status_str(status)} (status {status})")
        self.status = status


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the compiled library; raises if it has not been built."""
    global _lib
    if _lib is not None:  # loaded: no lock on the per-call path
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise ImportError(f"{path} is missing: build it with "
                                  "`python -m int4_weight_only_gemm_gb300._build`")
            lib = ctypes.CDLL(path)
            vp, sz, ci = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
            lib.w4a16_pack.argtypes = [vp, vp, ci, ci, vp]
            lib.w4a16_requant_pack.argtypes = [vp, vp, vp, ci, ci, ci, vp, vp]
            lib.w4a16_unpack.argtypes = [vp, vp, ci, ci, vp]
            lib.w4a16_pack_gate_up.argtypes = [vp, vp, ci, ci, vp]
            lib.w4a16_unpack_gate_up.argtypes = [vp, vp, ci, ci, vp]
            lib.w4a16_gemm_gate_up_silu.argtypes = [ci, ctypes.c_uint, vp, vp, vp, vp, ci, ci, ci, ci, vp, vp, sz, vp]
            lib.w4a16_workspace_bytes.argtypes = [ci, ci, ci, ci]
            lib.w4a16_workspace_bytes.restype = sz
            lib.w4a16_workspace_bytes_max.argtypes = [ci, ci, ci, ci]
            lib.w4a16_workspace_bytes_max.restype = sz
            lib.w4a16_workspace_bytes_path.argtypes = [ci, ci, ci, ci, ci]
            lib.w4a16_workspace_bytes_path.restype = sz
            lib.w4a16_set_workspace.argtypes = [vp, sz]
            lib.w4a16_gemm.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, vp, vp]
            lib.w4a16_gemm_ws.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, vp, vp, sz, vp]
            lib.w4a16_gemm_path.argtypes = [ci, vp, vp, vp, vp, ci, ci, ci, ci, vp, vp, sz, vp]
            lib.w4a16_gemm_ex.argtypes = [ci, ctypes.c_uint, vp, vp, vp, vp, ci, ci, ci, ci, vp, vp, sz, vp]
            lib.w4a16_auto_path.argtypes = [ci, ci, ci, ci]
            lib.w4a16_status_str.argtypes = [ci]
            lib.w4a16_status_str.restype = ctypes.c_char_p
            lib.w4a16_last_device_status.argtypes = [vp]
            lib.w4a16_launch_count.restype = ctypes.c_uint64
            lib.w4a16_swa_attention.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, ci, vp, vp, sz,
                                                ctypes.c_uint, vp]
            lib.w4a16_swa_workspace_bytes.argtypes = [ci, ci, ci, ci, ci, ci, ci]
            lib.w4a16_swa_workspace_bytes.restype = sz
            _lib = lib
    return _lib


# the current stream's handle without building a Stream object (a few
# microseconds a call); the public route where this torch lacks it
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device_index: int | None = None) -> int:
    if stream is None:
        if _raw_stream is not None:
            return int(_raw_stream(torch.cuda.current_device() if device_index is None else device_index))
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _raise(status: int, what: str):
    if status != W4A16_OK:
        raise W4A16Error(status, what)


def w4a16_status_str(status: int) -> str:
    return load_library().w4a16_status_str(int(status)).decode()


def w4a16_pack(qweight: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Canonical [K/8, N] int32 codes -> device layout (same size)."""
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    _check(qweight, "qweight", torch.int32)
    if out is None:
        out = torch.empty_like(qweight)
    _check(out, "out", torch.int32, qweight.shape)
    _raise(load_library().w4a16_pack(qweight.data_ptr(), out.data_ptr(), K, N, _stream(stream)), "w4a16_pack")
    return out


def w4a16_requant_pack(w: torch.Tensor, scales: torch.Tensor, qzeros: torch.Tensor, group: int = 128,
                       out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Re-quantize bf16 w [K, N] onto the frozen grid (scales, qzeros) straight
    into the device layout: code = clamp(round(w / s) + z, 0, 15)."""
    _check(w, "w", torch.bfloat16)
    if w.dim() != 2:
        raise ValueError("w must be [K, N]")
    K, N = w.shape
    G = K // group
    _check(scales, "scales", torch.float16, (G, N))
    _check(qzeros, "qzeros", torch.int32, (G, N // 8))
    if out is None:
        out = torch.empty((K // 8, N), dtype=torch.int32, device=w.device)
    _check(out, "out", torch.int32, (K // 8, N))
    _raise(load_library().w4a16_requant_pack(w.data_ptr(), scales.data_ptr(), qzeros.data_ptr(), K, N, group,
                                             out.data_ptr(), _stream(stream)), "w4a16_requant_pack")
    return out


def w4a16_unpack(qweight_dev: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Device layout -> canonical [K/8, N] int32 (exact inverse of w4a16_pack)."""
    _check(qweight_dev, "qweight_dev", torch.int32)
    K, N = qweight_dev.shape[0] * 8, qweight_dev.shape[1]
    if out is None:
        out = torch.empty_like(qweight_dev)
    _check(out, "out", torch.int32, qweight_dev.shape)
    _raise(load_library().w4a16_unpack(qweight_dev.data_ptr(), out.data_ptr(), K, N, _stream(stream)),
           "w4a16_unpack")
    return out


def w4a16_pack_gate_up(qweight: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Canonical [K/8, 2H] int32 codes of fused gate/up weights (gate columns
    first) -> the interleaved device layout of w4a16_gemm_gate_up_silu."""
    _check(qweight, "qweight", torch.int32)
    K, H = qweight.shape[0] * 8, qweight.shape[1] // 2
    if out is None:
        out = torch.empty_like(qweight)
    _check(out, "out", torch.int32, qweight.shape)
    _raise(load_library().w4a16_pack_gate_up(qweight.data_ptr(), out.data_ptr(), K, H, _stream(stream)),
           "w4a16_pack_gate_up")
    return out


def w4a16_unpack_gate_up(qweight_dev: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Exact inverse of w4a16_pack_gate_up."""
    _check(qweight_dev, "qweight_dev", torch.int32)
    K, H = qweight_dev.shape[0] * 8, qweight_dev.shape[1] // 2
    if out is None:
        out = torch.empty_like(qweight_dev)
    _check(out, "out", torch.int32, qweight_dev.shape)
    _raise(load_library().w4a16_unpack_gate_up(qweight_dev.data_ptr(), out.data_ptr(), K, H, _stream(stream)),
           "w4a16_unpack_gate_up")
    return out


def w4a16_gemm_gate_up_silu(x: torch.Tensor, qweight_dev: torch.Tensor, scales: torch.Tensor,
                            qzeros: torch.Tensor, group: int = 128, out: torch.Tensor | None = None,
                            workspace: torch.Tensor | None = None, path: int = PATH_AUTO, stream=None,
                            flags: int | None = None) -> torch.Tensor:
    """y = silu(x . Wg) * (x . Wu) in bf16 [M, H] for fused gate/up weights
    [K, 2H] packed by w4a16_pack_gate_up (scales / qzeros canonical, [G, 2H]
    and [G, 2H/8])."""
    _check(x, "x", torch.bfloat16)
    if x.dim() != 2:
        raise ValueError("x must be [M, K]")
    M, K = x.shape
    N = qweight_dev.shape[1]
    H = N // 2
    G = K // group if group > 0 else 0
    _check(qweight_dev, "qweight_dev", torch.int32, (K // 8, N))
    _check(scales, "scales", torch.float16, (G, N))
    _check(qzeros, "qzeros", torch.int32, (G, N // 8))
    if out is None:
        out = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
    _check(out, "out", torch.bfloat16, (M, H))
    lib = load_library()
    if workspace is None:
        need = _workspace_need(path, M, N, K, group, x.device)
        if need:
            workspace = _cached_workspace(need, x.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.w4a16_gemm_gate_up_silu(path, FLAG_PDL if flags is None else flags, x.data_ptr(),
                                     qweight_dev.data_ptr(), scales.data_ptr(), qzeros.data_ptr(), M, H, K, group,
                                     out.data_ptr(), ws_ptr, ws_bytes, _stream(stream))
    _raise(st, "w4a16_gemm_gate_up_silu")
    return out


def w4a16_workspace_bytes(M: int, N: int, K: int, group: int = 128, path: int = PATH_AUTO) -> int:
    return int(load_library().w4a16_workspace_bytes_path(path, M, N, K, group))


def w4a16_workspace_bytes_max(max_M: int, N: int, K: int, group: int = 128) -> int:
    return int(load_library().w4a16_workspace_bytes_max(max_M, N, K, group))


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled workspace buffer (the library needs it zeroed once)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def w4a16_set_workspace(workspace: torch.Tensor | None) -> None:
    lib = load_library()
    if workspace is None:
        _raise(lib.w4a16_set_workspace(None, 0), "w4a16_set_workspace")
    else:
        _raise(lib.w4a16_set_workspace(workspace.data_ptr(), workspace.numel() * workspace.element_size()),
               "w4a16_set_workspace")


_ws_cache: dict[int, torch.Tensor] = {}
_need_cache: dict[tuple, int] = {}


def _workspace_need(path: int, M: int, N: int, K: int, group: int, device: torch.device) -> int:
    """Workspace bytes a problem needs, asked of the library once per problem
    and device (the answer depends only on these)."""
    idx = device.index if device.index is not None else torch.cuda.current_device()
    key = (path, M, N, K, group, idx)
    need = _need_cache.get(key)
    if need is None:
        need = int(load_library().w4a16_workspace_bytes_path(path, M, N, K, group))
        _need_cache[key] = need
    return need


def _cached_workspace(nbytes: int, device: torch.device) -> torch.Tensor:
    idx = device.index if device.index is not None else torch.cuda.current_device()
    ws = _ws_cache.get(idx)
    if ws is None or ws.numel() < nbytes:
        ws = new_workspace(nbytes, device)
        _ws_cache[idx] = ws
    return ws


def w4a16_gemm(x: torch.Tensor, qweight_dev: torch.Tensor, scales: torch.Tensor, qzeros: torch.Tensor,
               group: int = 128, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
               path: int = PATH_AUTO, stream=None, flags: int | None = None) -> torch.Tensor:
    """y = x . dequant(qweight_dev, scales, qzeros) in bf16, on the GPU kernels.

    flags=None uses the library's default launch flags; otherwise a mask of
    FLAG_PDL and FLAG_STATIC_WEIGHTS (see include/w4a16.h)."""
    _check(x, "x", torch.bfloat16)
    if x.dim() != 2:
        raise ValueError("x must be [M, K]")
    M, K = x.shape
    N = qweight_dev.shape[1]
    G = K // group if group > 0 else 0
    _check(qweight_dev, "qweight_dev", torch.int32, (K // 8, N))
    _check(scales, "scales", torch.float16, (G, N))
    _check(qzeros, "qzeros", torch.int32, (G, N // 8))
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(out, "out", torch.bfloat16, (M, N))
    lib = load_library()
    if workspace is None:
        need = _workspace_need(path, M, N, K, group, x.device)
        if need:
            workspace = _cached_workspace(need, x.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    sp = _stream(stream, x.device.index)
    if flags is None:
        st = lib.w4a16_gemm_path(path, x.data_ptr(), qweight_dev.data_ptr(), scales.data_ptr(), qzeros.data_ptr(),
                                 M, N, K, group, out.data_ptr(), ws_ptr, ws_bytes, sp)
    else:
        st = lib.w4a16_gemm_ex(path, flags, x.data_ptr(), qweight_dev.data_ptr(), scales.data_ptr(),
                               qzeros.data_ptr(), M, N, K, group, out.data_ptr(), ws_ptr, ws_bytes, sp)
    _raise(st, "w4a16_gemm")
    return out


def w4a16_gemm_raw(x_ptr: int, qd_ptr: int, scales_ptr: int, qzeros_ptr: int, M: int, N: int, K: int,
                   group: int, y_ptr: int, ws_ptr: int | None, ws_bytes: int, path: int = PATH_AUTO,
                   stream: int = 0, flags: int | None = None) -> int:
    """Pointer-level call (no checks beyond the library's own), for timing loops."""
    lib = load_library()
    if flags is None:
        return lib.w4a16_gemm_path(path, x_ptr, qd_ptr, scales_ptr, qzeros_ptr, M, N, K, group, y_ptr,
                                   ws_ptr, ws_bytes, stream)
    return lib.w4a16_gemm_ex(path, flags, x_ptr, qd_ptr, scales_ptr, qzeros_ptr, M, N, K, group, y_ptr,
                             ws_ptr, ws_bytes, stream)


def w4a16_auto_path(M: int, N: int, K: int, group: int = 128) -> int:
    return int(load_library().w4a16_auto_path(M, N, K, group))


def w4a16_last_device_status(stream=None) -> int:
    return int(load_library().w4a16_last_device_status(_stream(stream)))


def w4a16_launch_count() -> int:
    return int(load_library().w4a16_launch_count())


def w4a16_swa_workspace_bytes(nq: int, Hq: int, Hkv: int, L: int, window: int, block: bool = False,
                              head_dim: int = 128) -> int:
    return int(load_library().w4a16_swa_workspace_bytes(nq, Hq, Hkv, head_dim, L, window, int(block)))


def w4a16_swa_attention(q: torch.Tensor, k_cache: torch.Tensor, vt_cache: torch.Tensor, L: int, window: int,
                        block: bool = False, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                        stream=None, flags: int = FLAG_PDL) -> torch.Tensor:
    """Sliding-window decode attention of a block of nq queries at positions
    L-nq .. L-1 (see include/w4a16.h).

    q [nq, Hq, 128] bf16; k_cache [Hkv, Lmax, 128] bf16; vt_cache [Hkv, 128,
    Lmax] bf16 (values transposed per head); returns out [nq, Hq, 128] bf16."""
    _check(q, "q", torch.bfloat16)
    _check(k_cache, "k_cache", torch.bfloat16)
    _check(vt_cache, "vt_cache", torch.bfloat16)
    if q.dim() != 3 or k_cache.dim() != 3 or vt_cache.dim() != 3:
        raise ValueError("q, k_cache, vt_cache must be 3-D")
    nq, Hq, d = q.shape
    Hkv, Lmax, _ = k_cache.shape
    if tuple(vt_cache.shape) != (Hkv, d, Lmax):
        raise ValueError(f"vt_cache has shape {tuple(vt_cache.shape)}, expected {(Hkv, d, Lmax)}")
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, q.shape)
    lib = load_library()
    need = int(lib.w4a16_swa_workspace_bytes(nq, Hq, Hkv, d, L, window, int(block)))
    if workspace is None:
        workspace = _cached_workspace(max(need, 1), q.device)
    st = lib.w4a16_swa_attention(q.data_ptr(), k_cache.data_ptr(), vt_cache.data_ptr(), nq, Hq, Hkv, d, L, Lmax,
                                 window, int(block), out.data_ptr(), workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(), flags, _stream(stream))
    _raise(st, "w4a16_swa_attention")
    return out


def to_device(problem, device="cuda"):
    """Host arrays of a w4a16_inputs.Problem -> CUDA tensors in the ABI dtypes."""
    import numpy as np
    x = torch.from_numpy(np.ascontiguousarray(problem.x).view(np.int16)).view(torch.bfloat16).to(device)
    qw = torch.from_numpy(np.ascontiguousarray(problem.qweight).view(np.int32)).to(device)
    sc = torch.from_numpy(np.ascontiguousarray(problem.scales).view(np.float16)).to(device)
    qz = torch.from_numpy(np.ascontiguousarray(problem.qzeros).view(np.int32)).to(device)
    return x, qw, sc, qz
