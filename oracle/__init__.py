"""CPU oracle for the W4A16 group-quantized GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its reference arm) may import this package.  The CUDA library and its
Python binding never do, and this package imports nothing from them.

Two independent renderings of the same plain definition
``y[m][n] = sum_k x[m][k] * (q[k][n] - z[k/g][n]) * s[k/g][n]`` (fp64):

* ``gemm`` / ``gemm_elems``: the C triple loop in ``w4a16_oracle.c``;
* ``gemm_numpy``: a numpy twin (fp64 dequantization, then ``numpy.matmul``),
  used as the library-routine cross-check on small inputs.

Sources: "Quantize the Target, Quantize the Drafter: Efficient Inference with
Qwen3.5-4B", pith.science review -- referee report summary (INT4 target with
its per-group scales kept) and "Assumptions & free parameters" (group size
128; packing rounds weights back onto the frozen per-group scales).  The
readings taken where the pages are silent (zero-point convention, nibble
order, zero packing along N, bf16/fp16 storage) are listed in the C file's
header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a16_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libw4a16_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP) into oracle/_build/."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u16p = ctypes.POINTER(ctypes.c_uint16)
            u32p = ctypes.POINTER(ctypes.c_uint32)
            u8p = ctypes.POINTER(ctypes.c_uint8)
            f64p = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            ci = ctypes.c_int
            lib.w4o_bf16_to_f64.restype = ctypes.c_double
            lib.w4o_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.w4o_f16_to_f64.restype = ctypes.c_double
            lib.w4o_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.w4o_f64_to_bf16_rne.restype = ctypes.c_uint16
            lib.w4o_f64_to_bf16_rne.argtypes = [ctypes.c_double]
            lib.w4o_pack_codes.argtypes = [u8p, ci, ci, u32p]
            lib.w4o_unpack_codes.argtypes = [u32p, ci, ci, u8p]
            lib.w4o_pack_zeros.argtypes = [u8p, ci, ci, u32p]
            lib.w4o_unpack_zeros.argtypes = [u32p, ci, ci, u8p]
            lib.w4o_dequant.argtypes = [u32p, u16p, u32p, ci, ci, ci, f64p]
            lib.w4o_gemm.argtypes = [u16p, u32p, u16p, u32p, ci, ci, ci, ci, f64p, ci]
            lib.w4o_gemm_elems.argtypes = [u16p, u32p, u16p, u32p, ci, ci, ci, ci,
                                           i64p, i64p, ctypes.c_int64, f64p, ci]
            lib.w4o_device_layout.argtypes = [u32p, ci, ci, u32p]
            lib.w4o_max_threads.restype = ci
            _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- scalar formats ---------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16)
    return np.array([lib.w4o_bf16_to_f64(int(v)) for v in b.ravel()]).reshape(b.shape)


def f16_to_f64(bits) -> np.ndarray:
    lib = _load()
    b = np.asarray(bits, dtype=np.uint16)
    return np.array([lib.w4o_f16_to_f64(int(v)) for v in b.ravel()]).reshape(b.shape)


def f64_to_bf16(vals) -> np.ndarray:
    lib = _load()
    v = np.asarray(vals, dtype=np.float64)
    return np.array([lib.w4o_f64_to_bf16_rne(float(a)) for a in v.ravel()],
                    dtype=np.uint16).reshape(v.shape)


# ---- packing ------------------------------------------------------------------

def pack_codes(codes: np.ndarray) -> np.ndarray:
    """codes[K][N] (0..15) -> canonical qweight[K/8][N] uint32."""
    codes = _c(codes, np.uint8)
    K, N = codes.shape
    out = np.zeros((K // 8, N), dtype=np.uint32)
    _load().w4o_pack_codes(_ptr(codes, ctypes.c_uint8), K, N, _ptr(out, ctypes.c_uint32))
    return out


def unpack_codes(qweight: np.ndarray) -> np.ndarray:
    qweight = _c(qweight, np.uint32)
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    out = np.zeros((K, N), dtype=np.uint8)
    _load().w4o_unpack_codes(_ptr(qweight, ctypes.c_uint32), K, N, _ptr(out, ctypes.c_uint8))
    return out


def pack_zeros(zeros: np.ndarray) -> np.ndarray:
    """zeros[G][N] (0..15) -> qzeros[G][N/8] uint32 (packed along N)."""
    zeros = _c(zeros, np.uint8)
    G, N = zeros.shape
    out = np.zeros((G, N // 8), dtype=np.uint32)
    _load().w4o_pack_zeros(_ptr(zeros, ctypes.c_uint8), G, N, _ptr(out, ctypes.c_uint32))
    return out


def unpack_zeros(qzeros: np.ndarray) -> np.ndarray:
    qzeros = _c(qzeros, np.uint32)
    G, N = qzeros.shape[0], qzeros.shape[1] * 8
    out = np.zeros((G, N), dtype=np.uint8)
    _load().w4o_unpack_zeros(_ptr(qzeros, ctypes.c_uint32), G, N, _ptr(out, ctypes.c_uint8))
    return out


def device_layout(qweight: np.ndarray) -> np.ndarray:
    """Canonical words -> the documented tiled device layout (flat uint32)."""
    qweight = _c(qweight, np.uint32)
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    if K % 128 or N % 8:
        raise ValueError("device layout needs K % 128 == 0 and N % 8 == 0")
    out = np.zeros(qweight.size, dtype=np.uint32)
    _load().w4o_device_layout(_ptr(qweight, ctypes.c_uint32), K, N, _ptr(out, ctypes.c_uint32))
    return out


# ---- dequantization and GEMM --------------------------------------------------

def dequant(qweight, scales, qzeros, group: int = 128) -> np.ndarray:
    qweight = _c(qweight, np.uint32)
    scales = _c(scales, np.uint16)
    qzeros = _c(qzeros, np.uint32)
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    W = np.zeros((K, N), dtype=np.float64)
    _load().w4o_dequant(_ptr(qweight, ctypes.c_uint32), _ptr(scales, ctypes.c_uint16),
                        _ptr(qzeros, ctypes.c_uint32), K, N, group, _ptr(W, ctypes.c_double))
    return W


def gemm(x, qweight, scales, qzeros, group: int = 128, nthreads: int = 0) -> np.ndarray:
    """Full y[M][N] in fp64 by the naive triple loop."""
    x = _c(x, np.uint16)
    qweight = _c(qweight, np.uint32)
    scales = _c(scales, np.uint16)
    qzeros = _c(qzeros, np.uint32)
    M, K = x.shape
    N = qweight.shape[1]
    assert qweight.shape[0] * 8 == K and scales.shape == (K // group, N)
    assert qzeros.shape == (K // group, N // 8)
    y = np.zeros((M, N), dtype=np.float64)
    _load().w4o_gemm(_ptr(x, ctypes.c_uint16), _ptr(qweight, ctypes.c_uint32),
                     _ptr(scales, ctypes.c_uint16), _ptr(qzeros, ctypes.c_uint32),
                     M, N, K, group, _ptr(y, ctypes.c_double), int(nthreads))
    return y


def gemm_elems(x, qweight, scales, qzeros, ms, ns, group: int = 128,
               nthreads: int = 0) -> np.ndarray:
    """Selected outputs y[ms[i]][ns[i]] in fp64, one by one."""
    x = _c(x, np.uint16)
    qweight = _c(qweight, np.uint32)
    scales = _c(scales, np.uint16)
    qzeros = _c(qzeros, np.uint32)
    ms = _c(ms, np.int64)
    ns = _c(ns, np.int64)
    M, K = x.shape
    N = qweight.shape[1]
    assert ms.shape == ns.shape
    if ms.size and (ms.min() < 0 or ms.max() >= M or ns.min() < 0 or ns.max() >= N):
        raise IndexError("sample index out of range")
    out = np.zeros(ms.shape, dtype=np.float64)
    _load().w4o_gemm_elems(_ptr(x, ctypes.c_uint16), _ptr(qweight, ctypes.c_uint32),
                           _ptr(scales, ctypes.c_uint16), _ptr(qzeros, ctypes.c_uint32),
                           M, N, K, group, _ptr(ms, ctypes.c_int64), _ptr(ns, ctypes.c_int64),
                           ms.size, _ptr(out, ctypes.c_double), int(nthreads))
    return out


def max_threads() -> int:
    return int(_load().w4o_max_threads())


# ---- numpy twin (independent second rendering, small inputs) -----------------

def _np_bf16(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gemm_numpy(x, qweight, scales, qzeros, group: int = 128) -> np.ndarray:
    """fp64 dequantization written with numpy array ops, then numpy.matmul."""
    qweight = np.asarray(qweight, dtype=np.uint32)
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    shifts = (4 * np.arange(8, dtype=np.uint32))[None, :, None]
    q = ((qweight[:, None, :] >> shifts) & 0xF).reshape(K, N).astype(np.float64)
    qz = np.asarray(qzeros, dtype=np.uint32)
    z = ((qz[:, :, None] >> shifts.reshape(1, 1, 8)) & 0xF).reshape(qz.shape[0], N)
    s = np.asarray(scales, dtype=np.uint16).view(np.float16).astype(np.float64)
    gidx = np.arange(K) // group
    W = (q - z[gidx].astype(np.float64)) * s[gidx]
    return np.matmul(_np_bf16(x), W)


def requant_codes(w, scales, qzeros, group: int = 128) -> np.ndarray:
    """Grid-preserving re-quantization: codes[k][n] = clamp(round(w / s) + z, 0, 15).

    The packing step of "Quantize the Target, Quantize the Drafter" (pith.science
    review, "Assumptions & free parameters": packing rounds the updated bf16
    weights back onto the frozen per-group scales; referee report summary: the
    model is re-packed onto the same grid).  w[K][N] are bf16 bits, scales
    [K/g][N] fp16 bits, qzeros [K/g][N/8] as for the GEMM; returns uint8 codes.

    The pages fix neither the rounding rule nor the precision of the quotient.
    Readings: round half to even, and the decision taken in IEEE binary32 --
    w and s are exact in binary32, w / s is the correctly rounded binary32
    quotient, rounded to the nearest integer (ties to even), z added, and the
    sum clipped to 0..15 -- the precision the CUDA kernel computes in.
    """
    w = np.asarray(w, dtype=np.uint16)
    K, N = w.shape
    G = K // group
    wf = bf16_to_f64(w).astype(np.float32)                       # exact
    sf = f16_to_f64(np.asarray(scales, dtype=np.uint16)).astype(np.float32)  # exact
    z = unpack_zeros(np.asarray(qzeros, dtype=np.uint32)).astype(np.float32)  # [G][N]
    gi = np.arange(K) // group                                   # group of row k
    quot = (wf / sf[gi, :]).astype(np.float32)                   # IEEE binary32 division
    r = np.rint(quot)                                            # nearest integer, ties to even
    c = np.clip(r + z[gi, :], 0.0, 15.0)
    assert c.shape == (K, N) and G * group == K
    return c.astype(np.uint8)


# ---- fused gate/up projection with the SiLU-multiply epilogue ----------------
#
# A gated MLP's gate and up projections stored as one weight matrix [K][2H]
# (gate columns 0..H-1, up columns H..2H-1) on one quantization grid, followed
# by y = silu(g) * u.  The pages name the fused gate/up shape of the decoder
# (2560 x 19456) but not the activation; the plain reading of a gated MLP is
# the one taken: silu(g) = g / (1 + exp(-g)) = g * logistic(g), applied to the
# exact products, so nothing is rounded before the final result.

def silu_mul(y: np.ndarray, H: int) -> np.ndarray:
    """y[:, :H] = gate pre-activations g, y[:, H:] = up values u -> g / (1 + e^-g) * u (fp64)."""
    y = np.asarray(y, dtype=np.float64)
    assert y.shape[-1] == 2 * H
    g, u = y[..., :H], y[..., H:]
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


def gemm_gate_up_silu(x, qweight, scales, qzeros, H: int, group: int = 128) -> np.ndarray:
    """Full silu(x . Wg) * (x . Wu) [M][H] in fp64: the triple-loop GEMM, then silu_mul."""
    return silu_mul(gemm(x, qweight, scales, qzeros, group), H)


def gemm_gate_up_silu_elems(x, qweight, scales, qzeros, H: int, ms, hs, group: int = 128) -> np.ndarray:
    """Selected outputs [ms[i]][hs[i]]: the gate and up products one by one, then silu * up."""
    ms = np.asarray(ms, dtype=np.int64)
    hs = np.asarray(hs, dtype=np.int64)
    g = gemm_elems(x, qweight, scales, qzeros, ms, hs, group)
    u = gemm_elems(x, qweight, scales, qzeros, ms, hs + H, group)
    return silu_mul(np.stack([g, u], axis=-1).reshape(-1, 2), 1).reshape(g.shape)


def gate_up_device_columns(H: int) -> np.ndarray:
    """canonical[d]: the canonical column held by device column d of the fused
    layout.  Each 128-column tile t holds 64 gate and 64 up columns; within the
    tile, block b of 16 columns holds gate columns 64t + 8b .. +7, then the up
    columns H + 64t + 8b .. +7."""
    d = np.arange(2 * H)
    t, j = d // 128, d % 128
    b, r = j // 16, j % 16
    return np.where(r < 8, 64 * t + 8 * b + r, H + 64 * t + 8 * b + (r - 8))


def device_layout_gate_up(qweight: np.ndarray, H: int) -> np.ndarray:
    """Canonical fused words [K/8][2H] -> device layout: the columns put in the
    interleaved order, then the plain tiled device layout."""
    qweight = _c(qweight, np.uint32)
    if H % 64 or qweight.shape[1] != 2 * H:
        raise ValueError("fused gate/up layout needs N = 2H with H % 64 == 0")
    return device_layout(np.ascontiguousarray(qweight[:, gate_up_device_columns(H)]))
