"""Pins of the fused gate/up oracle (CPU): the SiLU-multiply epilogue against
closed forms, an identity and a library routine, the half assignment, the
interleaved device column order, and the fused product against independent
renderings.

silu(g) = g / (1 + exp(-g)) applied to the gate half of a [K][2H] projection,
times the up half; the gated-MLP reading is stated in oracle/__init__.py.
"""
import numpy as np
import pytest

import oracle
import w4a16_inputs as wi


def test_silu_mul_hand_worked():
    # g = ln 3: 1 / (1 + 1/3) = 3/4, so silu(g) * 2 = 1.5 ln 3
    assert oracle.silu_mul(np.array([[np.log(3.0), 2.0]]), 1)[0, 0] == pytest.approx(1.5 * np.log(3.0), rel=1e-15)
    # g = 0 gives 0 whatever u is; g = ln(1/3): 1 / (1 + 3) = 1/4
    assert oracle.silu_mul(np.array([[0.0, 7.0]]), 1)[0, 0] == 0.0
    assert oracle.silu_mul(np.array([[-np.log(3.0), 4.0]]), 1)[0, 0] == pytest.approx(-np.log(3.0), rel=1e-15)


def test_silu_mul_matches_logistic_and_identity():
    scipy_special = pytest.importorskip("scipy.special")
    r = np.random.default_rng(3)
    g = r.uniform(-30, 30, 4000)
    u = r.standard_normal(4000)
    got = oracle.silu_mul(np.stack([g, u], axis=1), 1)[:, 0]
    np.testing.assert_allclose(got, g * scipy_special.expit(g) * u, rtol=1e-13, atol=1e-300)
    # silu(-g) = silu(g) - g
    ones = np.ones_like(g)
    s_pos = oracle.silu_mul(np.stack([g, ones], axis=1), 1)[:, 0]
    s_neg = oracle.silu_mul(np.stack([-g, ones], axis=1), 1)[:, 0]
    np.testing.assert_allclose(s_neg, s_pos - g, rtol=0, atol=1e-12)


def test_silu_mul_extremes_and_half_order():
    y = oracle.silu_mul(np.array([[-1000.0, 40.0, 3.0, 3.0]]), 2)
    assert np.all(np.isfinite(y)) and y[0, 0] == 0.0 and y[0, 1] == pytest.approx(120.0, rel=1e-15)
    # the first half is the gate: swapping the halves changes the result
    a = oracle.silu_mul(np.array([[2.0, 5.0]]), 1)[0, 0]
    b = oracle.silu_mul(np.array([[5.0, 2.0]]), 1)[0, 0]
    assert a == pytest.approx(2.0 / (1.0 + np.exp(-2.0)) * 5.0, rel=1e-15) and abs(a - b) > 1.0


def test_device_column_order():
    c = oracle.gate_up_device_columns(64)
    assert list(c[:24]) == list(range(0, 8)) + list(range(64, 72)) + list(range(8, 16))
    assert list(c[112:128]) == list(range(56, 64)) + list(range(120, 128))
    for H in (64, 128, 192, 9728):
        c = oracle.gate_up_device_columns(H)
        assert sorted(c.tolist()) == list(range(2 * H))  # a permutation
        # a gate column and its up column are 8 device columns apart, in one tile
        d = np.arange(2 * H)
        gate = d[(d % 16) < 8]
        assert np.array_equal(c[gate + 8], c[gate] + H)
        assert np.all(c[gate] // 64 == gate // 128)


def test_fused_product_against_numpy_rendering_and_samples():
    K, H, M = 256, 64, 5
    p = wi.generate(M, K, 2 * H, seed=21)
    full = oracle.gemm_gate_up_silu(p.x, p.qweight, p.scales, p.qzeros, H)
    twin = oracle.silu_mul(oracle.gemm_numpy(p.x, p.qweight, p.scales, p.qzeros), H)
    np.testing.assert_allclose(full, twin, rtol=1e-12, atol=1e-12)
    ms = np.array([0, 1, 4, 4, 2])
    hs = np.array([0, 63, 5, 40, 17])
    np.testing.assert_allclose(oracle.gemm_gate_up_silu_elems(p.x, p.qweight, p.scales, p.qzeros, H, ms, hs),
                               full[ms, hs], rtol=1e-14, atol=1e-14)


def test_fused_one_hot_closed_form():
    # x = e_k: g = (q[k][h] - z) s and u = (q[k][H+h] - z') s', so y = silu(g) u exactly
    K, H = 128, 64
    p = wi.generate(1, K, 2 * H, seed=22)
    k = 37
    x = np.zeros((1, K), dtype=np.uint16)
    x[0, k] = 0x3F80  # 1.0 in bf16
    codes = oracle.unpack_codes(p.qweight).astype(np.float64)
    z = oracle.unpack_zeros(p.qzeros).astype(np.float64)
    s = oracle.f16_to_f64(p.scales)
    g = (codes[k, :H] - z[0, :H]) * s[0, :H]
    u = (codes[k, H:] - z[0, H:]) * s[0, H:]
    want = g / (1.0 + np.exp(-g)) * u
    np.testing.assert_allclose(oracle.gemm_gate_up_silu(x, p.qweight, p.scales, p.qzeros, H)[0], want,
                               rtol=1e-15, atol=1e-15)


# ---- the pins above catch plausible mistakes in the epilogue (planted here, on the CPU) ----

def _pins_hold(silu_mul):
    """The hand-worked, identity and half-order pins, applied to a candidate rendering."""
    ok = abs(silu_mul(np.array([[np.log(3.0), 2.0]]), 1)[0, 0] - 1.5 * np.log(3.0)) < 1e-12
    g = np.linspace(-8, 8, 33)
    ones = np.ones_like(g)
    s_pos = silu_mul(np.stack([g, ones], axis=1), 1)[:, 0]
    s_neg = silu_mul(np.stack([-g, ones], axis=1), 1)[:, 0]
    ok = ok and np.allclose(s_neg, s_pos - g, atol=1e-12)
    ok = ok and abs(silu_mul(np.array([[2.0, 5.0]]), 1)[0, 0] - 2.0 / (1.0 + np.exp(-2.0)) * 5.0) < 1e-12
    return bool(ok)


def _halves(y, H):
    y = np.asarray(y, dtype=np.float64)
    return y[..., :H], y[..., H:]


MUTANTS = {
    "halves swapped": lambda y, H: (lambda g, u: u / (1.0 + np.exp(-u)) * g)(*_halves(y, H)),
    "exp sign": lambda y, H: (lambda g, u: g / (1.0 + np.exp(g)) * u)(*_halves(y, H)),
    "sigmoid only": lambda y, H: (lambda g, u: 1.0 / (1.0 + np.exp(-g)) * u)(*_halves(y, H)),
    "no gate factor": lambda y, H: (lambda g, u: g * u)(*_halves(y, H)),
    "tanh gate": lambda y, H: (lambda g, u: g * 0.5 * (1.0 + np.tanh(g)) * u)(*_halves(y, H)),
}


def test_pins_hold_for_the_oracle():
    assert _pins_hold(oracle.silu_mul)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_a_planted_mistake(name):
    assert not _pins_hold(MUTANTS[name]), f"the pins miss the mistake: {name}"
