"""Pins of the sliding-window decode attention oracle (oracle/swa.py) against
facts the definition fixes, independent of the oracle's own formula:

* a one-key window returns that key's value exactly;
* equal scores (q = 0) give the plain mean of the window's values;
* keys outside a query's window have no effect, keys inside it do;
* two keys: the weights are the logistic function of the score difference
  (scipy.special.expit), with the 1/sqrt(d) scale;
* grouped-query heads: with each key/value head's values constant, query head
  h returns the constant of head h // (Hq / Hkv);
* a dominant score selects its value (the sign of the exponent);
* the block form: every query of the block sees the same window.

"Quantize the Target, Quantize the Drafter" (pith.science review,
"Assumptions & free parameters": SWA window 1024 / 2048, DFlash block 16).
A second group plants plausible mistakes in a copy of the definition and
checks that the pins catch each one.
"""
import numpy as np
import pytest
from scipy.special import expit

import w4a16_inputs as wi
from oracle import swa


def bf16(a):
    return wi.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def dec(bits):
    return swa._bf16(bits)


def rand(shape, seed, scale=1.0):
    r = np.random.default_rng(seed)
    return bf16(r.standard_normal(shape) * scale)


def test_window_bounds():
    lo, hi = swa.window_bounds(L=10, nq=3, W=4)
    assert lo.tolist() == [4, 5, 6] and hi.tolist() == [7, 8, 9]
    lo, hi = swa.window_bounds(L=3, nq=3, W=8)          # window longer than the context
    assert lo.tolist() == [0, 0, 0] and hi.tolist() == [0, 1, 2]
    lo, hi = swa.window_bounds(L=10, nq=3, W=4, block=True)
    assert lo.tolist() == [6, 6, 6] and hi.tolist() == [9, 9, 9]


def pins(attn):
    """Every pin, run against an implementation `attn(q, k, v, W, block)`."""
    d, Hq, Hkv, L, nq = 8, 4, 2, 12, 3
    q, k, v = rand((nq, Hq, d), 1), rand((Hkv, L, d), 2), rand((Hkv, L, d), 3)
    # one-key window: that key's value, exactly
    out = attn(q, k, v, 1, False)
    for i in range(nq):
        for h in range(Hq):
            assert np.array_equal(out[i, h], dec(v)[h // 2, L - nq + i])
    # equal scores: the mean of the window's values
    W = 5
    out = attn(np.zeros_like(q), k, v, W, False)
    for i in range(nq):
        e = L - nq + i
        want = dec(v)[:, e - W + 1:e + 1].mean(axis=1)
        for h in range(Hq):
            assert np.allclose(out[i, h], want[h // 2], rtol=0, atol=1e-12)
    # outside the window: no effect; inside: an effect
    base = attn(q, k, v, W, False)
    k2, v2 = k.copy(), v.copy()
    k2[:, :L - nq - W + 1] = rand((Hkv, L - nq - W + 1, d), 9)
    v2[:, :L - nq - W + 1] = rand((Hkv, L - nq - W + 1, d), 10)
    assert np.array_equal(attn(q, k2, v2, W, False)[0], base[0])
    v3 = v.copy()
    v3[:, L - nq - W + 1] = bf16(dec(v[:, L - nq - W + 1]) + 1.0)  # first key of query 0's window
    assert not np.allclose(attn(q, k, v3, W, False)[0], base[0])
    v4 = v.copy()
    v4[:, L - 1] = bf16(dec(v[:, L - 1]) + 1.0)                     # a later block token: causal
    assert np.array_equal(attn(q, k, v4, W, False)[0], base[0])
    assert not np.allclose(attn(q, k, v4, W, True)[0], attn(q, k, v, W, True)[0])
    # two keys: logistic weights of the scaled score difference
    out = attn(q[:1], k[:, :2], v[:, :2], 2, False)
    qq, kk, vv = dec(q[:1]), dec(k[:, :2]), dec(v[:, :2])
    for h in range(Hq):
        s = kk[h // 2] @ qq[0, h] / np.sqrt(d)
        w1 = expit(s[1] - s[0])
        want = (1 - w1) * vv[h // 2, 0] + w1 * vv[h // 2, 1]
        assert np.allclose(out[0, h], want, rtol=1e-12, atol=1e-12)
    # grouped-query heads: constant values per key/value head
    vc = np.stack([np.full((L, d), c, np.float32) for c in (0.5, -2.0)])
    out = attn(q, k, bf16(vc), W, False)
    for h in range(Hq):
        assert np.allclose(out[:, h], [0.5, -2.0][h // 2], rtol=0, atol=1e-12)
    # a dominant score selects its value
    kd = np.zeros((Hkv, L, d), np.float32)
    kd[:, L - 2, 0] = 1.0
    qd = np.zeros((nq, Hq, d), np.float32)
    qd[:, :, 0] = 64.0
    out = attn(bf16(qd), bf16(kd), v, W, False)
    for h in range(Hq):
        assert np.allclose(out[nq - 1, h], dec(v)[h // 2, L - 2], atol=1e-6)
    # block form: every query sees the same window
    out = attn(np.repeat(q[:1], nq, axis=0), k, v, W, True)
    assert np.array_equal(out[0], out[nq - 1])


def test_oracle_satisfies_pins():
    pins(swa.swa_attention)


def test_oracle_at_full_head_shape():
    """32 query heads over 8 key/value heads of width 128, a window of 1024 and
    a 16-token block: finite, and each output is a convex combination of the
    window's values (within their per-coordinate range)."""
    nq, Hq, Hkv, d, L, W = 16, 32, 8, 128, 1100, 1024
    q, k, v = rand((nq, Hq, d), 4), rand((Hkv, L, d), 5), rand((Hkv, L, d), 6)
    out = swa.swa_attention(q, k, v, W)
    assert out.shape == (nq, Hq, d) and np.all(np.isfinite(out))
    vv = dec(v)
    lo, hi = swa.window_bounds(L, nq, W)
    for i in (0, nq - 1):
        win = vv[:, lo[i]:hi[i] + 1]
        for h in (0, Hq - 1):
            assert np.all(out[i, h] <= win[h // 4].max(axis=0) + 1e-12)
            assert np.all(out[i, h] >= win[h // 4].min(axis=0) - 1e-12)


# ---- planted mistakes: each must fail the pins --------------------------------

def _planted(kind):
    def attn(q, k, v, W, block=False):
        q, k, v = dec(q), dec(k), dec(v)
        nq, Hq, d = q.shape
        Hkv, L, _ = k.shape
        g = Hq // Hkv
        out = np.zeros((nq, Hq, d))
        for i in range(nq):
            e = L - 1 if block else L - nq + i
            lo = max(0, e - W + 1)
            if kind == "window_one_short":
                lo = max(0, e - W + 2) if W > 1 else lo
            if kind == "window_one_long":
                lo = max(0, e - W)
            hi = e + 1
            if kind == "sees_whole_block":
                hi = L
            for h in range(Hq):
                hk = h % Hkv if kind == "head_modulo" else h // g
                s = k[hk, lo:hi] @ q[i, h]
                s = s * np.sqrt(d) if kind == "scale_sqrt_d" else s / np.sqrt(d)
                if kind == "exp_sign":
                    s = -s
                p = np.exp(s - s.max())
                o = p @ v[hk, lo:hi]
                out[i, h] = o if kind == "no_normalisation" else o / p.sum()
        return out
    return attn


@pytest.mark.parametrize("kind", ["window_one_short", "window_one_long", "sees_whole_block", "head_modulo",
                                  "scale_sqrt_d", "exp_sign", "no_normalisation"])
def test_pins_catch_planted_mistake(kind):
    with pytest.raises(AssertionError):
        pins(_planted(kind))


def test_planted_copy_without_mistake_passes():
    pins(_planted("none"))
