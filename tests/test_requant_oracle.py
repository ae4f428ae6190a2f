"""Pins of the oracle's grid-preserving re-quantization (CPU only):
codes[k][n] = clamp(round(w / s) + z, 0, 15), round half to even, decided in
IEEE binary32 ("Quantize the Target, Quantize the Drafter", pith.science
review, "Assumptions & free parameters": packing rounds the updated bf16
weights back onto the frozen per-group scales)."""
from fractions import Fraction

import numpy as np

import oracle
import w4a16_inputs as wi


def _w(vals):
    return wi.f32_to_bf16_bits(np.asarray(vals, dtype=np.float32))


def _s(vals):
    return wi.f64_to_f16_bits(np.asarray(vals, dtype=np.float64))


def _z(vals):
    return oracle.pack_zeros(np.asarray(vals, dtype=np.uint8))


def test_hand_worked():
    # w = 4.0, s = 0.5, z = 3: 4 / 0.5 = 8, + 3 = 11
    c = oracle.requant_codes(_w(np.full((128, 8), 4.0)), _s(np.full((1, 8), 0.5)), _z(np.full((1, 8), 3)))
    assert (c == 11).all()


def test_ties_go_to_even():
    vals = [-2.5, -1.5, -0.5, 0.5, 1.5, 2.5, 3.5, 4.5]
    w = np.zeros((128, 8), dtype=np.float32)
    w[0, :] = vals
    c = oracle.requant_codes(_w(w), _s(np.ones((1, 8))), _z(np.full((1, 8), 8)))
    assert c[0].tolist() == [6, 6, 8, 8, 10, 10, 12, 12]


def test_clipped_to_the_code_range():
    w = np.zeros((128, 8), dtype=np.float32)
    w[0, :] = [100.0, -100.0, 12.0, -3.0, -4.0, 11.0, 12.4, -3.4]
    c = oracle.requant_codes(_w(w), _s(np.ones((1, 8))), _z(np.full((1, 8), 3)))
    assert c[0].tolist() == [15, 0, 15, 0, 0, 14, 15, 0]


def test_row_k_uses_group_k_div_128():
    # w = 1/16 everywhere; group 0 has s = 1/64, group 1 s = 1/32, z = 0
    w = np.full((256, 8), 1.0 / 16, dtype=np.float32)
    s = np.array([[1 / 64] * 8, [1 / 32] * 8])
    c = oracle.requant_codes(_w(w), _s(s), _z(np.zeros((2, 8))))
    assert (c[:128] == 4).all() and (c[128:] == 2).all()


def test_round_trip_through_dequant():
    """bf16(dequant(q)) re-quantizes to q: the bf16 rounding moves w by at most
    15 s / 512 < s / 2, so the nearest grid point is the original one."""
    rng = np.random.default_rng(11)
    K, N = 384, 64
    codes = rng.integers(0, 16, (K, N), dtype=np.uint8)
    zeros = rng.integers(0, 16, (K // 128, N), dtype=np.uint8)
    scales = _s(rng.uniform(0.001, 0.02, (K // 128, N)))
    qw, qz = oracle.pack_codes(codes), oracle.pack_zeros(zeros)
    w = oracle.f64_to_bf16(oracle.dequant(qw, scales, qz))
    assert (oracle.requant_codes(w, scales, qz) == codes).all()


def test_against_exact_rationals():
    """Brute force: the exact quotient rounded half to even, except where it
    lies within 1e-6 of a half-integer (there binary32 may decide either way)."""
    rng = np.random.default_rng(12)
    K, N = 128, 16
    w = _w(rng.standard_normal((K, N)).astype(np.float32) * 0.05)
    s = _s(rng.uniform(0.001, 0.02, (1, N)))
    zeros = rng.integers(0, 16, (1, N), dtype=np.uint8)
    got = oracle.requant_codes(w, s, _z(zeros))
    wv = oracle.bf16_to_f64(w)
    sv = oracle.f16_to_f64(s)
    checked = 0
    for k in range(K):
        for n in range(N):
            q = Fraction(float(wv[k, n])) / Fraction(float(sv[0, n]))
            fl = q.numerator // q.denominator
            frac = q - fl
            if abs(float(frac) - 0.5) < 1e-6:
                continue
            r = fl + 1 if frac > Fraction(1, 2) else fl
            want = min(15, max(0, r + int(zeros[0, n])))
            assert got[k, n] == want, (k, n)
            checked += 1
    assert checked > K * N * 0.99
