"""Pins for the W4A16 GEMM oracle: checks against facts that do not come from
the oracle itself (hand-worked values, closed forms, exact rational
arithmetic, integer special cases that reduce to an integer matmul).

Each pin takes a GEMM implementation ``impl(x, qweight, scales, qzeros, group)``
returning fp64 ``y[M][N]`` and raises AssertionError when it disagrees.  The
oracle must pass every pin (tests/test_oracle.py); deliberately broken
variants of the definition must each fail at least one (tests/test_pins_catch.py).

The definition pinned: y[m][n] = sum_k x[m][k] * (q[k][n] - z[k/g][n]) * s[k/g][n]
with codes packed low-nibble-first along K and zeros packed along N
("Quantize the Target, Quantize the Drafter", pith.science review: INT4
weights with per-group scales, group size 128).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

G128 = 128


def _pack_k(codes: np.ndarray) -> np.ndarray:
    """Independent canonical packer for test construction (numpy shifts)."""
    codes = np.asarray(codes, dtype=np.uint32)
    K, N = codes.shape
    c = codes.reshape(K // 8, 8, N)
    return np.bitwise_or.reduce(c << (4 * np.arange(8, dtype=np.uint32))[None, :, None], axis=1).astype(np.uint32)


def _pack_n(zeros: np.ndarray) -> np.ndarray:
    zeros = np.asarray(zeros, dtype=np.uint32)
    G, N = zeros.shape
    z = zeros.reshape(G, N // 8, 8)
    return np.bitwise_or.reduce(z << (4 * np.arange(8, dtype=np.uint32))[None, None, :], axis=2).astype(np.uint32)


def _bf16_bits(vals) -> np.ndarray:
    """Exactly representable values -> bfloat16 bits via float32 truncation."""
    f = np.asarray(vals, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bfloat16"
    return (u >> 16).astype(np.uint16)


def _f16_bits(vals) -> np.ndarray:
    h = np.asarray(vals, dtype=np.float64).astype(np.float16)
    assert np.all(h.astype(np.float64) == np.asarray(vals, dtype=np.float64))
    return h.view(np.uint16)


def _rng(seed):
    return np.random.default_rng(seed)


# ---- pins ------------------------------------------------------------------

def pin_zero_codes_zero_points(impl):
    """All codes 0 with all zero points 0 give y = 0 whatever x and s are."""
    r = _rng(1)
    K, N, M = 256, 16, 3
    x = _bf16_bits(r.integers(-8, 8, size=(M, K)))
    q = np.zeros((K, N), np.uint8)
    z = np.zeros((K // G128, N), np.uint8)
    s = _f16_bits(r.integers(1, 64, size=(K // G128, N)) / 64.0)
    y = impl(x, _pack_k(q), s, _pack_n(z), G128)
    assert np.all(y == 0.0), "zero codes and zero points must give y = 0"


def pin_q_equals_z(impl):
    """Codes equal to their group's zero point give y = 0."""
    r = _rng(2)
    K, N, M = 384, 24, 2
    z = r.integers(0, 16, size=(K // G128, N)).astype(np.uint8)
    q = np.repeat(z, G128, axis=0)
    x = (r.standard_normal((M, K)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    s =_f16_bits(r.integers(1, 1000, size=(K // G128, N)) / 1024.0)
    y = impl(x, _pack_k(q), s, _pack_n(z), G128)
    assert np.all(y == 0.0), "q == z must give y = 0"


def pin_unit_scale_offset8(impl):
    """s = 1, z = 8: y = x . (q - 8), checked against an int64 matmul."""
    r = _rng(3)
    K, N, M = 256, 40, 4
    xi = r.integers(-100, 101, size=(M, K))
    q = r.integers(0, 16, size=(K, N))
    x = _bf16_bits(xi)
    s = _f16_bits(np.ones((K // G128, N)))
    z = np.full((K // G128, N), 8, np.uint8)
    y = impl(x, _pack_k(q), s, _pack_n(z), G128)
    want = xi.astype(np.int64) @ (q.astype(np.int64) - 8)
    assert np.array_equal(y, want.astype(np.float64)), "s=1, z=8 must give x.(q-8)"


def pin_one_hot_rows(impl):
    """x = e_k picks row k of the dequantized matrix: y[n] = (q[k][n]-z[k/g][n]) s[k/g][n]."""
    r = _rng(4)
    K, N = 384, 16
    q = r.integers(0, 16, size=(K, N))
    z = r.integers(0, 16, size=(K // G128, N))
    sv = r.integers(1, 2048, size=(K // G128, N)) * 2.0 ** -14
    ks = np.array([0, 1, 7, 8, 127, 128, 200, 255, 256, 383])
    xv = np.zeros((len(ks), K))
    xv[np.arange(len(ks)), ks] = 1.0
    y = impl(_bf16_bits(xv), _pack_k(q), _f16_bits(sv), _pack_n(z), G128)
    for i, k in enumerate(ks):
        g = k // G128
        want = np.array([(int(q[k, n]) - int(z[g, n])) * Fraction(sv[g, n]) for n in range(N)],
                        dtype=object)
        got = y[i]
        assert all(Fraction(float(got[n])) == want[n] for n in range(N)), f"one-hot row {k}"


def pin_group_sums(impl):
    """x = 1 on the rows of group j, 0 elsewhere: y[n] = s[j][n] (sum_k q[k][n] - 128 z[j][n])."""
    K, N = 384, 8
    k = np.arange(K)[:, None]
    n = np.arange(N)[None, :]
    q = (k * 3 + n * 5) % 16
    z = (np.arange(K // G128)[:, None] * 7 + np.arange(N)[None, :] * 2) % 16
    sv = (1 + np.arange(K // G128)[:, None] * N + np.arange(N)[None, :]) * 2.0 ** -10
    xv = np.zeros((K // G128, K))
    for j in range(K // G128):
        xv[j, j * G128:(j + 1) * G128] = 1.0
    y = impl(_bf16_bits(xv), _pack_k(q), _f16_bits(sv), _pack_n(z), G128)
    for j in range(K // G128):
        colsum = q[j * G128:(j + 1) * G128].sum(axis=0)
        want = sv[j] * (colsum - 128 * z[j])
        assert np.array_equal(y[j], want), f"group {j} sums"


def pin_hand_worked(impl):
    """Hand-worked K=128, N=8, M=1 example (tests/golden/hand_worked_k128.txt).

    x = 1 for every k; q[k][n] = (k + n) mod 16, so each column's codes run
    through 0..15 eight times and sum to 960; z[n] = n; s[n] = 2^-(n+1).
    Then y[n] = 2^-(n+1) (960 - 128 n) = 480, 208, 88, 36, 14, 5, 1.5, 0.25.
    """
    K, N = 128, 8
    k = np.arange(K)[:, None]
    n = np.arange(N)[None, :]
    q = (k + n) % 16
    z = np.arange(N)[None, :]
    s = 2.0 ** -(np.arange(N)[None, :] + 1)
    y = impl(_bf16_bits(np.ones((1, K))), _pack_k(q), _f16_bits(s), _pack_n(z), G128)
    assert np.array_equal(y[0], [480.0, 208.0, 88.0, 36.0, 14.0, 5.0, 1.5, 0.25]), y


def pin_exact_rational(impl):
    """Brute force with exact rationals on random tiny problems.

    Inputs are decoded through numpy's IEEE float16/float32 (a different
    route from the oracle's own bit-field decoding), the sum is exact, and
    the fp64 result must agree to within the fp64 accumulation error bound.
    """
    r = _rng(5)
    for (M, K, N) in [(2, 128, 8), (1, 256, 16), (3, 256, 8)]:
        G = K // G128
        qw = r.integers(0, 1 << 32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32)
        qz = r.integers(0, 1 << 32, size=(G, N // 8), dtype=np.uint64).astype(np.uint32)
        s = r.uniform(0.001, 0.02, size=(G, N)).astype(np.float16)
        xf = r.standard_normal((M, K)).astype(np.float32)
        xb = (xf.view(np.uint32) >> 16).astype(np.uint16)  # truncation: any bf16 is fine
        y = impl(xb, qw, s.view(np.uint16), qz, G128)
        xv = (xb.astype(np.uint32) << 16).view(np.float32)
        for m in range(M):
            for n in range(N):
                acc = Fraction(0)
                absacc = Fraction(0)
                for kk in range(K):
                    qv = (int(qw[kk // 8, n]) >> (4 * (kk % 8))) & 0xF
                    zv = (int(qz[kk // G128, n // 8]) >> (4 * (n % 8))) & 0xF
                    t = Fraction(float(xv[m, kk])) * (qv - zv) * Fraction(float(s[kk // G128, n]))
                    acc += t
                    absacc += abs(t)
                err = abs(Fraction(float(y[m, n])) - acc)
                assert err <= absacc * K * Fraction(2) ** -52, (m, n, float(err))


def pin_linearity(impl):
    """y(x1 + x2) = y(x1) + y(x2) exactly when every sum is exact in fp64."""
    r = _rng(6)
    K, N, M = 256, 16, 3
    x1 = r.integers(-64, 64, size=(M, K))
    x2 = r.integers(-64, 64, size=(M, K))
    qw = r.integers(0, 1 << 32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32)
    qz = r.integers(0, 1 << 32, size=(K // G128, N // 8), dtype=np.uint64).astype(np.uint32)
    s = _f16_bits(r.integers(1, 256, size=(K // G128, N)) * 2.0 ** -8)
    ya = impl(_bf16_bits(x1), qw, s, qz, G128)
    yb = impl(_bf16_bits(x2), qw, s, qz, G128)
    yc = impl(_bf16_bits(x1 + x2), qw, s, qz, G128)
    assert np.array_equal(ya + yb, yc), "linearity in x"


def pin_columns_independent(impl):
    """Changing one column's codes, zero or scale changes only that column."""
    r = _rng(7)
    K, N, M = 256, 16, 2
    q = r.integers(0, 16, size=(K, N))
    z = r.integers(0, 16, size=(K // G128, N))
    sv = r.integers(1, 512, size=(K // G128, N)) * 2.0 ** -12
    x = _bf16_bits(r.integers(-4, 5, size=(M, K)))
    y0 = impl(x, _pack_k(q), _f16_bits(sv), _pack_n(z), G128)
    for col in (0, 5, 9, 15):
        q2, z2, s2 = q.copy(), z.copy(), sv.copy()
        q2[:, col] = (q2[:, col] + 3) % 16
        z2[1, col] = (z2[1, col] + 1) % 16
        s2[0, col] *= 2
        y1 = impl(x, _pack_k(q2), _f16_bits(s2), _pack_n(z2), G128)
        other = [c for c in range(N) if c != col]
        assert np.array_equal(y0[:, other], y1[:, other]), f"column {col} leaked"
        assert not np.array_equal(y0[:, col], y1[:, col])


ALL_PINS = [
    pin_zero_codes_zero_points,
    pin_q_equals_z,
    pin_unit_scale_offset8,
    pin_one_hot_rows,
    pin_group_sums,
    pin_hand_worked,
    pin_exact_rational,
    pin_linearity,
    pin_columns_independent,
]
