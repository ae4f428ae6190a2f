"""CPU oracle for sliding-window decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module; the CUDA library and its binding never do, and
this module imports nothing from them.

What it computes (the plain definition, fp64, no blocking or reordering):
the drafter's attention restricted to a sliding window of W keys, for a block
of nq query tokens appended at the end of a context of L tokens.

    e_i   = L - nq + i      (causal: query i sees itself and what precedes it)
          = L - 1           (block: every query of the block sees the whole block)
    J_i   = { j : max(0, e_i - W + 1) <= j <= e_i }
    s_ij  = (q[i, h] . k[hk, j]) / sqrt(d)                   for j in J_i
    out[i, h] = sum_{j in J_i} exp(s_ij - max_J s) v[hk, j] / sum_{j in J_i} exp(s_ij - max_J s)

with grouped-query heads: query head h reads key/value head hk = h // (Hq / Hkv).

Sources: "Quantize the Target, Quantize the Drafter: Efficient Inference with
Qwen3.5-4B" -- pith.science review, "Assumptions & free parameters" (SWA
window length 1024 on the leaderboard, 1024 or 2048 after the latency /
acceptance trade-off; DFlash block size 16) and referee summary (the 5-layer
block-diffusion drafter is equipped with sliding-window attention); the
gptget.net summary's key results (sliding-window attention reduces
long-context decoding latency); the Longformer entry of the mlsanity.com
"builds on" list (the sliding-window pattern).

Readings where the pages are silent:
  - the window holds the W most recent positions up to and including the
    query's own (Longformer's one-sided, causal form);
  - scores are scaled by 1/sqrt(d), the usual dot-product attention;
  - heads: the width of the layer's attention output (4096 = the o_proj K of
    the decoder shapes) gives Hq = 32 query heads of d = 128; the key/value
    heads are Hkv = 8 (grouped-query, 4 query heads per key/value head);
  - the block of nq = 16 draft tokens is causal by default; ``block=True``
    lets every draft token see the whole block (a block-diffusion drafter
    denoises its block jointly), with the same window length;
  - q, k, v are bfloat16, decoded exactly; everything after is fp64.
"""
from __future__ import annotations

import numpy as np


def _bf16(bits) -> np.ndarray:
    """bfloat16 bits -> fp64 (exact: a bfloat16 is the top half of a binary32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def window_bounds(L: int, nq: int, W: int, block: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """First and last visible key position of each query of the block."""
    i = np.arange(nq)
    e = np.full(nq, L - 1) if block else L - nq + i
    lo = np.maximum(0, e - W + 1)
    return lo, e


def swa_attention(q, k, v, W: int, block: bool = False) -> np.ndarray:
    """q [nq][Hq][d], k and v [Hkv][L][d] (bfloat16 bits) -> out [nq][Hq][d] fp64.

    Query i, head h: softmax over keys j in its window of q.k / sqrt(d), then
    the weighted sum of the values, one query and one head at a time.
    """
    q, k, v = _bf16(q), _bf16(k), _bf16(v)
    nq, Hq, d = q.shape
    Hkv, L, _ = k.shape
    assert Hq % Hkv == 0 and v.shape == k.shape and nq <= L
    group = Hq // Hkv
    lo, hi = window_bounds(L, nq, W, block)
    out = np.zeros((nq, Hq, d), dtype=np.float64)
    for i in range(nq):
        for h in range(Hq):
            hk = h // group
            keys = k[hk, lo[i]:hi[i] + 1]            # [n][d]
            vals = v[hk, lo[i]:hi[i] + 1]
            s = keys @ q[i, h] / np.sqrt(d)          # scores
            p = np.exp(s - s.max())                  # unnormalised weights
            out[i, h] = (p @ vals) / p.sum()
    return out
