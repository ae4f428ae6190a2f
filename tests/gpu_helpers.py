"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
(via the thin binding) and compare with the CPU oracle.

Tolerance (applied element by element and in aggregate):
    |y_gpu - y_ref| <= 1e-2 * (|y_ref| + 1)   and   ||y_gpu - y_ref||_F / ||y_ref||_F <= 5e-3
where y_ref is the oracle's fp64 result and y_gpu the kernel's bfloat16 output.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import w4a16_inputs as wi

ELEM_RTOL = 1e-2
FRO_TOL = 5e-3


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def check_close(y_gpu: np.ndarray, y_ref: np.ndarray, what: str = ""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert y_gpu.shape == y_ref.shape, (y_gpu.shape, y_ref.shape)
    assert np.all(np.isfinite(y_gpu)), f"{what}: non-finite output"
    err = np.abs(y_gpu - y_ref)
    bound = ELEM_RTOL * (np.abs(y_ref) + 1.0)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance, e.g. "
                             + ", ".join(f"{tuple(i)} gpu={y_gpu[tuple(i)]:.6g} ref={y_ref[tuple(i)]:.6g}"
                                         for i in idx))
    nref = np.linalg.norm(y_ref)
    fro = np.linalg.norm(y_gpu - y_ref) / nref if nref > 0 else np.linalg.norm(y_gpu)
    assert fro <= FRO_TOL, f"{what}: relative Frobenius error {fro:.3e} > {FRO_TOL}"
    return float(fro), float(err.max())


class Device:
    """A problem resident on the GPU in the ABI's formats, packed once."""

    def __init__(self, prob: wi.Problem):
        import int4_weight_only_gemm_gb300 as w
        self.w = w
        self.prob = prob
        self.x, self.qw, self.scales, self.qzeros = w.to_device(prob)
        self.qd = w.w4a16_pack(self.qw)

    def run(self, path=0, x=None, workspace=None, flags=None, out=None) -> torch.Tensor:
        x = self.x if x is None else x
        return self.w.w4a16_gemm(x, self.qd, self.scales, self.qzeros, path=path, workspace=workspace,
                                 flags=flags, out=out)


def sample_indices(M: int, N: int, count: int, seed: int):
    """Random (m, n) pairs plus the four corners and the last row and column."""
    r = np.random.default_rng(seed)
    ms = r.integers(0, M, count)
    ns = r.integers(0, N, count)
    extra_m = np.array([0, 0, M - 1, M - 1] + [M - 1] * 8 + list(r.integers(0, M, 8)))
    extra_n = np.array([0, N - 1, 0, N - 1] + list(r.integers(0, N, 8)) + [N - 1] * 8)
    return np.concatenate([ms, extra_m]), np.concatenate([ns, extra_n])


def check_sampled(dev: Device, y: torch.Tensor, count: int = 3000, seed: int = 0, what: str = ""):
    p = dev.prob
    ms, ns = sample_indices(p.M, p.N, count, seed)
    ref = oracle.gemm_elems(p.x, p.qweight, p.scales, p.qzeros, ms, ns)
    got = bf16_to_f64(y[torch.as_tensor(ms, device=y.device), torch.as_tensor(ns, device=y.device)])
    return check_close(got, ref, what)
