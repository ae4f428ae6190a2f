"""Seeded synthetic inputs for the W4A16 group-quantized GEMM.

This module is the only code shared by the CPU oracle side (tests, golden-value
scripts, the CPU baseline) and the CUDA side (tests, benchmark).  It holds no
arithmetic of the method itself: it draws random bits and encodes random reals
into the storage formats the GEMM consumes, nothing else.

Workload source: "Quantize the Target, Quantize the Drafter: Efficient Inference
with Qwen3.5-4B" (pith.science review, "Assumptions & free parameters": GPTQ
group size 128 for the INT4 drafter; referee summary: AWQ INT4 target with
per-group scales; "DFlash block size 16" sets the 16-token verify block).  The
pages print no tensor, so the values below are synthetic stand-ins with the
layer shapes of a ~4B decoder:

* packed codes ``qweight[K/8][N]`` (uint32): every bit uniform, so each of the
  eight 4-bit codes in a word is an independent uniform draw from 0..15;
* zero points ``qzeros[K/128][N/8]`` (uint32): likewise, one uniform 4-bit zero
  per (group, column);
* scales ``scales[K/128][N]``: uniform on [0.001, 0.02] drawn in float64 and
  rounded to IEEE binary16 (round to nearest even); returned as uint16 bits;
* activations ``x[M][K]``: float32 standard normal rounded to bfloat16 (round
  to nearest even); returned as uint16 bits.

Generator: ``numpy.random.Generator(PCG64(SeedSequence([seed, shape_idx, M])))``
with draw order qweight, qzeros, scales, x.
"""
from __future__ import annotations

import dataclasses

import numpy as np

GROUP = 128

# (K, N) of the four projections of one decoder layer, plus the vocabulary head.
SHAPES = {
    "qkv": (2560, 4096),
    "o_proj": (4096, 2560),
    "gate_up": (2560, 19456),
    "down": (9728, 2560),
    "vocab": (2560, 151936),
}
SHAPE_INDEX = {"qkv": 0, "o_proj": 1, "gate_up": 2, "down": 3, "vocab": 4}
LAYER = ("qkv", "o_proj", "gate_up", "down")

# Workloads by name: (seed, list of (shape name, M)).
WORKLOADS = {
    "tiny": (0, [("tiny", 1)]),
    "decode_m1": (1, [(s, 1) for s in LAYER]),
    "verify_m16": (2, [(s, 16) for s in LAYER]),
    "prefill_m2048": (3, [(s, 2048) for s in LAYER]),
    "sweep": (4, [(s, m) for m in (1, 2, 4, 8, 16, 32, 64, 128, 8192) for s in LAYER]
              + [("vocab", 1), ("vocab", 16)]),
}
TINY = (256, 128)


def shape_kn(name: str) -> tuple[int, int]:
    return TINY if name == "tiny" else SHAPES[name]


def shape_idx(name: str) -> int:
    return 0 if name == "tiny" else SHAPE_INDEX[name]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); uint16 bits.

    Inputs are finite by construction here (normal draws), so no NaN handling.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def f64_to_f16_bits(a: np.ndarray) -> np.ndarray:
    """Round float64 values to IEEE binary16 (numpy's cast rounds to nearest even)."""
    return np.asarray(a, dtype=np.float64).astype(np.float16).view(np.uint16)


@dataclasses.dataclass
class Problem:
    """One GEMM problem in the storage formats of the public interface."""

    M: int
    K: int
    N: int
    group: int
    x: np.ndarray        # [M][K] uint16 (bfloat16 bits)
    qweight: np.ndarray  # [K/8][N] uint32, canonical packing
    scales: np.ndarray   # [K/group][N] uint16 (binary16 bits)
    qzeros: np.ndarray   # [K/group][N/8] uint32

    @property
    def G(self) -> int:
        return self.K // self.group


def generate(M: int, K: int, N: int, seed: int, shape_index: int = 0,
             group: int = GROUP, rng_key: tuple | None = None) -> Problem:
    """Draw one problem from the seeded recipe described in the module docstring."""
    if K % group or K % 8 or N % 8:
        raise ValueError("K must divide by the group and by 8, N by 8")
    key = list(rng_key) if rng_key is not None else [seed, shape_index, M]
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(key)))
    G = K // group
    qweight = rng.integers(0, 1 << 32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32)
    qzeros = rng.integers(0, 1 << 32, size=(G, N // 8), dtype=np.uint64).astype(np.uint32)
    scales = f64_to_f16_bits(rng.uniform(0.001, 0.02, size=(G, N)))
    x = f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    return Problem(M, K, N, group, x, qweight, scales, qzeros)


def generate_named(shape: str, M: int, seed: int) -> Problem:
    K, N = shape_kn(shape)
    return generate(M, K, N, seed, shape_idx(shape))


def random_x(M: int, K: int, seed: int) -> np.ndarray:
    """Extra activation rows (bfloat16 bits) from an independent stream."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0xA11, M, K])))
    return f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))


def random_weights(K: int, N: int, seed: int, sigma: float = 0.05) -> np.ndarray:
    """Dense weights w[K][N] (bfloat16 bits) for the re-quantization step:
    float32 normal draws with standard deviation `sigma`, rounded to bfloat16
    (nearest, ties to even).  With scales in [0.001, 0.02], w / s spans well
    past the 0..15 code range, so clipping is exercised too."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x5EC, K, N])))
    return f32_to_bf16_bits(rng.standard_normal((K, N), dtype=np.float32) * np.float32(sigma))
