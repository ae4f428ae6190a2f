"""GPU parity of the sliding-window decode attention kernel (w4a16_swa_attention,
through the C ABI) against the fp64 oracle (oracle/swa.py).

Workloads follow "Quantize the Target, Quantize the Drafter" (pith.science
review, "Assumptions & free parameters": SWA window 1024 / 2048, DFlash block
of 16; the scenarios' 64/128, 2048/256 and 8192/256 input/output tokens give
the context lengths): 32 query heads over 8 key/value heads of width 128,
q, k, v ~ N(0, 1) rounded to bf16, seeded.

Tolerance, from the arithmetic (scores and softmax in f32, the weights
rounded once to bf16 for the product with v, the result rounded to bf16):
per element |gpu - ref| <= 1e-2 |ref| + 4e-3 rms(v), and relative Frobenius
error <= 5e-3.
"""
import numpy as np
import pytest
import torch

import w4a16_inputs as wi
from oracle import swa

pytestmark = pytest.mark.gpu


def make(nq, Hq, Hkv, L, Lmax, seed):
    r = np.random.default_rng(seed)
    q = wi.f32_to_bf16_bits(r.standard_normal((nq, Hq, 128), dtype=np.float32))
    k = wi.f32_to_bf16_bits(r.standard_normal((Hkv, Lmax, 128), dtype=np.float32))
    v = wi.f32_to_bf16_bits(r.standard_normal((Hkv, Lmax, 128), dtype=np.float32))
    return q, k, v


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def run(q, k, v, L, W, block, ws=None):
    import int4_weight_only_gemm_gb300 as w
    vt = np.ascontiguousarray(np.transpose(v, (0, 2, 1)))  # [Hkv][128][Lmax]
    out = w.w4a16_swa_attention(dev(q), dev(k), dev(vt), L, W, block, workspace=ws)
    torch.cuda.synchronize()
    return out


def check(out, q, k, v, L, W, block, what):
    ref = swa.swa_attention(q, k[:, :L], v[:, :L], W, block)
    got = out.float().cpu().numpy().astype(np.float64)
    vv = swa._bf16(v[:, :L])
    rms = float(np.sqrt(np.mean(vv * vv)))
    err = np.abs(got - ref)
    bound = 1e-2 * np.abs(ref) + 4e-3 * rms
    assert np.all(np.isfinite(got)), what
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} out of tolerance, max err {err.max():.3g}"
    fro = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert fro <= 5e-3, f"{what}: relative Frobenius {fro:.3g}"


# (nq, Hq, Hkv, L, Lmax, W, block): the scenarios' context lengths with both windows
CASES = [
    (16, 32, 8, 192, 192, 1024, False),     # short prompt: the window covers everything
    (16, 32, 8, 2304, 2304, 1024, False),   # medium
    (16, 32, 8, 2304, 2304, 2048, False),
    (16, 32, 8, 8448, 8448, 1024, False),   # long
    (16, 32, 8, 8448, 8448, 2048, True),    # block form
    (1, 32, 8, 8448, 8448, 2048, False),    # one query (plain decode)
    (1, 32, 8, 100, 104, 1024, False),
    (3, 8, 2, 37, 40, 16, False),           # ragged L, short window
    (32, 32, 8, 700, 704, 300, False),      # 128 query rows, a window that is no multiple of 8
    (5, 4, 4, 64, 64, 1, False),            # one-key window, one head per group
    (7, 12, 3, 1000, 1000, 64, True),
]


@pytest.mark.parametrize("nq,Hq,Hkv,L,Lmax,W,block", CASES)
def test_swa_matches_oracle(nq, Hq, Hkv, L, Lmax, W, block):
    q, k, v = make(nq, Hq, Hkv, L, Lmax, seed=nq * 1000 + L + W)
    out = run(q, k, v, L, W, block)
    check(out, q, k, v, L, W, block, f"nq={nq} Hq={Hq} Hkv={Hkv} L={L} W={W} block={block}")


def test_swa_deterministic_and_workspace_reused():
    import int4_weight_only_gemm_gb300 as w
    q, k, v = make(16, 32, 8, 3000, 3000, seed=7)
    ws = w.new_workspace(w.w4a16_swa_workspace_bytes(16, 32, 8, 3000, 2048))
    a = run(q, k, v, 3000, 2048, False, ws)
    b = run(q, k, v, 3000, 2048, False, ws)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    n0 = w.w4a16_launch_count()
    run(q, k, v, 3000, 2048, False, ws)
    assert w.w4a16_launch_count() == n0 + 2  # the chunk kernel and the combine
    assert w.w4a16_last_device_status() == 0


def test_swa_keys_past_L_are_not_read():
    """Positions L..Lmax-1 of the caches hold NaN: the result must not see them."""
    q, k, v = make(4, 8, 2, 300, 400, seed=11)
    k[:, 300:] = 0x7FC0
    v[:, 300:] = 0x7FC0
    out = run(q, k, v, 300, 128, False)
    check(out, q, k, v, 300, 128, False, "NaN past L")


def test_swa_argument_errors():
    import int4_weight_only_gemm_gb300 as w
    lib = w.load_library()
    q = torch.zeros((2, 8, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((2, 64, 128), dtype=torch.bfloat16, device="cuda")
    vt = torch.zeros((2, 128, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    ws = w.new_workspace(1 << 20)

    def call(nq=2, Hq=8, Hkv=2, d=128, L=64, Lmax=64, W=16, block=0, flags=1, wsb=1 << 20):
        return lib.w4a16_swa_attention(q.data_ptr(), kc.data_ptr(), vt.data_ptr(), nq, Hq, Hkv, d, L, Lmax, W, block,
                                       out.data_ptr(), ws.data_ptr(), wsb, flags, 0)
    assert call() == 0
    assert call(d=64) == w.W4A16_EUNSUPPORTED
    assert call(Hkv=3) == w.W4A16_EINVAL           # Hq % Hkv
    assert call(L=65) == w.W4A16_EINVAL            # L > Lmax
    assert call(Lmax=60) == w.W4A16_EINVAL         # Lmax % 8
    assert call(W=0) == w.W4A16_EINVAL
    assert call(nq=40) == w.W4A16_EUNSUPPORTED    # 160 query rows per head group
    assert call(flags=2) == w.W4A16_EINVAL
    assert call(wsb=16) == w.W4A16_EWORKSPACE
    torch.cuda.synchronize()
    assert w.w4a16_last_device_status() == 0


def test_swa_shares_a_workspace_with_the_gemm():
    """One buffer as the workspace of the attention and of a split-K GEMM: the
    attention leaves the GEMM's arrival counters (the first 64 KB) at zero."""
    import int4_weight_only_gemm_gb300 as w
    import oracle
    from tests.gpu_helpers import Device, bf16_to_f64, check_close
    p = wi.generate_named("qkv", 1, 60)
    d = Device(p)
    q, k, v = make(16, 32, 8, 2304, 2304, seed=61)
    need = max(w.w4a16_workspace_bytes(1, p.N, p.K, path=w.PATH_GEMV_SPLITK),
               w.w4a16_swa_workspace_bytes(16, 32, 8, 2304, 1024))
    ws = w.new_workspace(need)
    for _ in range(2):
        run(q, k, v, 2304, 1024, False, ws)
        assert ws[:65536].view(torch.int32).abs().sum().item() == 0
        y = d.run(w.PATH_GEMV_SPLITK, workspace=ws)
        torch.cuda.synchronize()
        check_close(bf16_to_f64(y), oracle.gemm(p.x, p.qweight, p.scales, p.qzeros), "split-K after attention")
