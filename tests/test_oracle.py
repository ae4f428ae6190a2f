"""The CPU oracle against its pins (no GPU needed).

Sources for what is pinned: "Quantize the Target, Quantize the Drafter:
Efficient Inference with Qwen3.5-4B", pith.science review -- referee report
summary (INT4 AWQ target, per-group scales frozen, weights re-packed on the
same grid) and "Assumptions & free parameters" (group size 128).
"""
import os

import numpy as np
import pytest

import oracle
import w4a16_inputs as wi
from tests import oracle_pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _impl(x, qw, s, qz, group):
    return oracle.gemm(x, qw, s, qz, group)


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(_impl)


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_numpy_twin_pin(pin):
    pin(oracle.gemm_numpy)


# ---- number formats -----------------------------------------------------------

def test_bf16_decode_all_values():
    """Every bfloat16 pattern decodes to the float32 whose top half it is."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    want = (bits << 16).view(np.float32).astype(np.float64)
    got = oracle.bf16_to_f64(bits.astype(np.uint16))
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_f16_decode_all_values():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = oracle.f16_to_f64(bits)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_bf16_decode_hand_values():
    assert oracle.bf16_to_f64(np.uint16(0x3F80)) == 1.0
    assert oracle.bf16_to_f64(np.uint16(0xC000)) == -2.0
    assert oracle.bf16_to_f64(np.uint16(0x4300)) == 128.0
    assert oracle.bf16_to_f64(np.uint16(0x430F)) == 143.0
    assert oracle.bf16_to_f64(np.uint16(0x0001)) == 2.0 ** -133
    assert oracle.bf16_to_f64(np.uint16(0x0080)) == 2.0 ** -126


def test_bf16_round_hand_values():
    # ties go to the even significand
    assert oracle.f64_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle.f64_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert oracle.f64_to_bf16(-(1.0 + 2.0 ** -8 + 2.0 ** -30)) == 0xBF81
    assert oracle.f64_to_bf16(255.5) == 0x4380          # 255.5 -> 256 (tie, even)
    assert oracle.f64_to_bf16(0.0) == 0x0000
    assert oracle.f64_to_bf16(-0.0) == 0x8000
    assert oracle.f64_to_bf16(2.0 ** -133) == 0x0001
    assert oracle.f64_to_bf16(3.0 * 2.0 ** 127 * 2) == 0x7F80  # overflow -> inf


def test_bf16_round_is_nearest_even():
    """RNE against brute force over the neighbouring bfloat16 values."""
    r = np.random.default_rng(11)
    vals = np.concatenate([r.standard_normal(2000) * 10.0 ** r.integers(-30, 30, 2000),
                           r.standard_normal(500) * 2.0 ** -128])
    out = oracle.f64_to_bf16(vals)
    dec = oracle.bf16_to_f64(out)
    for v, b, d in zip(vals, out, dec):
        nbrs = oracle.bf16_to_f64(np.array([(int(b) - 1) & 0xFFFF, (int(b) + 1) & 0xFFFF], np.uint16))
        for nb in nbrs:
            if np.sign(nb) == np.sign(d) or nb == 0:
                assert abs(v - d) <= abs(v - nb), (v, hex(b))
                if abs(v - d) == abs(v - nb):
                    assert int(b) % 2 == 0


# ---- packing --------------------------------------------------------------------

def test_pack_hand_worked():
    """K=8, N=1, codes 0..7 -> 0x76543210 (low nibble = row 0)."""
    codes = np.arange(8, dtype=np.uint8).reshape(8, 1)
    assert oracle.pack_codes(codes)[0, 0] == 0x76543210
    zeros = np.arange(8, dtype=np.uint8).reshape(1, 8)
    assert oracle.pack_zeros(zeros)[0, 0] == 0x76543210


def test_pack_unpack_roundtrip():
    r = np.random.default_rng(12)
    for codes in (r.integers(0, 16, size=(256, 40)), np.zeros((64, 8), int),
                  np.full((64, 8), 15), (np.arange(128)[:, None] + np.arange(24)[None, :]) % 16):
        codes = codes.astype(np.uint8)
        qw = oracle.pack_codes(codes)
        assert np.array_equal(oracle.unpack_codes(qw), codes)
        assert np.array_equal(qw, oracle_pins._pack_k(codes))
    z = r.integers(0, 16, size=(5, 64)).astype(np.uint8)
    assert np.array_equal(oracle.unpack_zeros(oracle.pack_zeros(z)), z)


def test_dequant_hand_worked():
    """q=11, z=3, s=0.5 -> 4.0; s=1, z=8 -> q-8; q=z -> 0."""
    K, N = 128, 8
    codes = np.full((K, N), 11, np.uint8)
    zeros = np.full((1, N), 3, np.uint8)
    s = np.full((1, N), 0.5, np.float16).view(np.uint16)
    W = oracle.dequant(oracle.pack_codes(codes), s, oracle.pack_zeros(zeros))
    assert np.all(W == 4.0)
    codes = (np.arange(K)[:, None] % 16 + np.zeros((1, N), int)).astype(np.uint8)
    W = oracle.dequant(oracle.pack_codes(codes), np.full((1, N), 1.0, np.float16).view(np.uint16),
                       oracle.pack_zeros(np.full((1, N), 8, np.uint8)))
    assert np.array_equal(W, codes.astype(np.float64) - 8)


def test_device_layout_hand_worked():
    """One word: canonical nibbles r=0..7 (0x76543210) land at positions
    p = [0,2,4,6,1,3,5,7] -> 0x75316420; its position for column 0 is word 0."""
    K, N = 128, 8
    qw = np.zeros((K // 8, N), np.uint32)
    qw[0, 0] = 0x76543210
    d = oracle.device_layout(qw)
    assert d[0] == 0x75316420 and np.count_nonzero(d) == 1
    # word row kw = 4c + j, column t  ->  (c*W + t)*4 + j with W = 8
    qw = np.zeros((K // 8, N), np.uint32)
    qw[6, 3] = 0x11111111                      # kw = 6 -> c = 1, j = 2
    d = oracle.device_layout(qw)
    assert np.flatnonzero(d).tolist() == [(1 * 8 + 3) * 4 + 2]


def test_device_layout_is_permutation():
    r = np.random.default_rng(13)
    for (K, N) in [(256, 128), (384, 264), (128, 8)]:
        qw = r.integers(0, 1 << 32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32)
        d = oracle.device_layout(qw)
        assert d.size == qw.size
        # every canonical word appears exactly once, nibbles re-ordered
        nib = [(qw >> (4 * r)) & 0xF for r in range(8)]
        order = [0, 2, 4, 6, 1, 3, 5, 7]
        perm = np.zeros_like(qw)
        for p, r_ in enumerate(order):
            perm |= nib[r_] << (4 * p)
        assert np.array_equal(np.sort(d), np.sort(perm.ravel()))
        # a word whose nibbles are all equal is unchanged by the re-order,
        # so a per-column constant lands in that column's positions only
        col = np.broadcast_to((np.arange(N, dtype=np.uint32) % 15 + 1) * 0x11111111, qw.shape)
        dc = oracle.device_layout(np.ascontiguousarray(col))
        W0 = min(128, N)
        assert np.all(dc[: W0 * 16].reshape(4, W0, 4)[:, :, :] ==
                      ((np.arange(W0, dtype=np.uint32) % 15 + 1) * 0x11111111)[None, :, None])


# ---- oracle internals vs each other ------------------------------------------

def test_numpy_twin_agrees_on_configs():
    for shape, M, seed in [("tiny", 1, 0), ("qkv", 2, 1)]:
        p = wi.generate_named(shape, M, seed)
        if shape != "tiny":  # keep it small: trim to a column slice
            p = wi.Problem(M, p.K, 256, 128, p.x, p.qweight[:, :256].copy(),
                           p.scales[:, :256].copy(), p.qzeros[:, :32].copy())
        y = oracle.gemm(p.x, p.qweight, p.scales, p.qzeros)
        y2 = oracle.gemm_numpy(p.x, p.qweight, p.scales, p.qzeros)
        assert np.max(np.abs(y - y2)) <= 1e-12 * max(1.0, np.max(np.abs(y)))


def test_elems_match_full_and_threads_deterministic():
    p = wi.generate(5, 512, 264, seed=9)
    y1 = oracle.gemm(p.x, p.qweight, p.scales, p.qzeros, nthreads=1)
    y4 = oracle.gemm(p.x, p.qweight, p.scales, p.qzeros, nthreads=4)
    assert np.array_equal(y1, y4)
    r = np.random.default_rng(0)
    ms = r.integers(0, 5, 50)
    ns = r.integers(0, 264, 50)
    ye = oracle.gemm_elems(p.x, p.qweight, p.scales, p.qzeros, ms, ns)
    assert np.array_equal(ye, y1[ms, ns])


def test_other_group_sizes():
    """The definition is the same for any group size dividing K."""
    r = np.random.default_rng(14)
    for g in (32, 64, 256):
        K, N, M = 512, 16, 2
        qw = r.integers(0, 1 << 32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32)
        qz = r.integers(0, 1 << 32, size=(K // g, N // 8), dtype=np.uint64).astype(np.uint32)
        s = r.uniform(0.001, 0.02, size=(K // g, N)).astype(np.float16).view(np.uint16)
        x = wi.f32_to_bf16_bits(r.standard_normal((M, K)).astype(np.float32))
        y = oracle.gemm(x, qw, s, qz, g)
        y2 = oracle.gemm_numpy(x, qw, s, qz, g)
        assert np.max(np.abs(y - y2)) <= 1e-12 * np.max(np.abs(y))


def test_golden_hand_worked_fixture():
    """tests/golden/hand_worked_k128.txt holds the hand-derived outputs."""
    vals = _read_golden(os.path.join(GOLDEN, "hand_worked_k128.txt"))
    assert vals == [480.0, 208.0, 88.0, 36.0, 14.0, 5.0, 1.5, 0.25]
    oracle_pins.pin_hand_worked(_impl)


def test_golden_tiny_config_fixture():
    """tests/golden/tiny_m1_k256_n128.txt was written by tests/golden/make_golden.py
    (which calls only the oracle); the oracle must still reproduce it bit for bit."""
    vals = _read_golden(os.path.join(GOLDEN, "tiny_m1_k256_n128.txt"))
    p = wi.generate_named("tiny", 1, 0)
    y = oracle.gemm(p.x, p.qweight, p.scales, p.qzeros)
    assert np.array_equal(np.array(vals), y[0])


def _read_golden(path):
    out = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            out.append(float.fromhex(line) if "0x" in line else float(line))
    return out
