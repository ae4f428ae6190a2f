"""GPU parity of the W4A16 GEMM (through the C ABI) against the CPU oracle.

Workloads are the seeded synthetic problems of w4a16_inputs: the tiny case,
the decode set (M=1) and verify set (M=16) over the four projection shapes of
a ~4B decoder layer, prefill (M=2048), the M sweep up to 8192 and the
vocabulary-shaped GEMM ("Quantize the Target, Quantize the Drafter":
pith.science review -- INT4 target and drafter, group size 128, DFlash block
size 16).  Every problem is compared in full, except M=8192, where at least
256 whole rows are (every row of the first and last token tiles and one row
of every other tile).  Both kernels (GEMV and tensor core) are checked at
every M either can run.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import w4a16_inputs as wi
from tests.gpu_helpers import Device, bf16_bits, bf16_to_f64, check_close, check_sampled

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GEMV, TC, AUTO, SPLITK, CS = 1, 2, 0, 3, 4
GEMV_FORMS = [SPLITK, CS]  # the GEMV's two forms, forced


def _full(prob, y, what):
    ref = oracle.gemm(prob.x, prob.qweight, prob.scales, prob.qzeros)
    return check_close(bf16_to_f64(y), ref, what)


# ---- config 0: tiny -----------------------------------------------------------

@pytest.mark.parametrize("path", [AUTO, GEMV, TC])
def test_tiny_config(path):
    p = wi.generate_named("tiny", 1, 0)
    d = Device(p)
    y = d.run(path)
    _full(p, y, f"tiny path={path}")
    # stored values written by tests/golden/make_golden.py from the oracle
    vals = [float.fromhex(l) for l in open(os.path.join(GOLDEN, "tiny_m1_k256_n128.txt"))
            if l.strip() and not l.startswith("#")]
    check_close(bf16_to_f64(y)[0], np.array(vals), "tiny vs golden")


# ---- config 1 / 2: decode (M=1) and verify (M=16) sets, in full ---------------

@pytest.mark.parametrize("shape", wi.LAYER)
@pytest.mark.parametrize("path", [AUTO, GEMV, TC, SPLITK, CS])
def test_decode_set_m1(shape, path):
    p = wi.generate_named(shape, 1, 1)
    y = Device(p).run(path)
    _full(p, y, f"decode {shape} path={path}")


@pytest.mark.parametrize("shape", wi.LAYER)
def test_verify_set_m16(shape):
    p = wi.generate_named(shape, 16, 2)
    y = Device(p).run(AUTO)
    _full(p, y, f"verify {shape}")


# ---- config 3: prefill M=2048, in full ------------------------------------------

@pytest.mark.parametrize("shape", wi.LAYER)
def test_prefill_m2048_full(shape):
    """Every output of the four projections at M=2048.  For the gate_up shape
    the same oracle product also checks the fused gate/up kernel: the weights
    are packed by w4a16_pack_gate_up and y = silu(gate) * up."""
    import int4_weight_only_gemm_gb300 as w
    p = wi.generate_named(shape, 2048, 3)
    d = Device(p)
    ref = oracle.gemm(p.x, p.qweight, p.scales, p.qzeros)
    check_close(bf16_to_f64(d.run(AUTO)), ref, f"prefill {shape}")
    if shape == "gate_up":
        H = p.N // 2
        qd = w.w4a16_pack_gate_up(d.qw)
        y = w.w4a16_gemm_gate_up_silu(d.x, qd, d.scales, d.qzeros)
        check_close(bf16_to_f64(y), oracle.silu_mul(ref, H), "prefill fused gate_up")


# ---- config 4: M sweep and the vocabulary shape ------------------------------

@pytest.mark.parametrize("M", [2, 4, 8])
@pytest.mark.parametrize("shape", wi.LAYER)
def test_sweep_small_m_both_paths(M, shape):
    p = wi.generate_named(shape, M, 4)
    d = Device(p)
    ref = oracle.gemm(p.x, p.qweight, p.scales, p.qzeros)
    for path in (GEMV, TC, SPLITK, CS):
        check_close(bf16_to_f64(d.run(path)), ref, f"sweep {shape} M={M} path={path}")


@pytest.mark.parametrize("M", [16, 32, 48])  # 48: three 16-token draft blocks verified together
@pytest.mark.parametrize("shape", wi.LAYER)
def test_sweep_mid_m_full(M, shape):
    p = wi.generate_named(shape, M, 4)
    _full(p, Device(p).run(AUTO), f"sweep {shape} M={M}")


@pytest.mark.parametrize("M", [64, 128])
@pytest.mark.parametrize("shape", wi.LAYER)
def test_sweep_large_m_full(M, shape):
    _full(*_run_auto(shape, M, 4), f"sweep {shape} M={M}")


def _run_auto(shape, M, seed):
    p = wi.generate_named(shape, M, seed)
    return p, Device(p).run(AUTO)


def rows_m8192(M=8192, seed=8192):
    """Whole rows checked at M=8192: every row of the first and the last
    192-token tile, one seeded row from every other tile, and seeded rows
    beyond those to make up at least 256."""
    nt = 192
    tiles = (M + nt - 1) // nt
    r = np.random.default_rng(seed)
    rows = set(range(0, nt)) | set(range((tiles - 1) * nt, M))
    rows |= {int(t * nt + r.integers(0, nt)) for t in range(1, tiles - 1)}
    while len(rows) < 400:
        rows.add(int(r.integers(0, M)))
    return np.array(sorted(rows))


@pytest.mark.parametrize("shape", wi.LAYER)
def test_sweep_m8192_whole_rows(shape):
    p, y = _run_auto(shape, 8192, 4)
    rows = rows_m8192()
    assert len(rows) >= 256
    ref = oracle.gemm(np.ascontiguousarray(p.x[rows]), p.qweight, p.scales, p.qzeros)
    check_close(bf16_to_f64(y[torch.as_tensor(rows, device=y.device)]), ref, f"sweep {shape} M=8192 rows")


@pytest.mark.parametrize("M,path", [(1, GEMV), (1, SPLITK), (1, TC), (16, TC)])
def test_vocab_shape_full(M, path):
    p = wi.generate_named("vocab", M, 4)
    _full(p, Device(p).run(path), f"vocab M={M} path={path}")


# ---- edge cases: ragged tiles, odd M, one group --------------------------------

EDGE = [(M, K, N) for (K, N) in [(128, 8), (128, 136), (384, 264), (1024, 392)]
        for M in (1, 3, 7, 13, 17, 31, 33, 100, 129, 257, 400)]


@pytest.mark.parametrize("M,K,N", EDGE)
def test_ragged_and_odd_shapes(M, K, N):
    p = wi.generate(M, K, N, seed=M * 7 + K + N)
    d = Device(p)
    ref = oracle.gemm(p.x, p.qweight, p.scales, p.qzeros)
    paths = [SPLITK, CS, TC] if M <= 8 else [TC]
    for path in paths:
        check_close(bf16_to_f64(d.run(path)), ref, f"M={M} K={K} N={N} path={path}")


@pytest.mark.parametrize("M", [1, 5, 16, 40, 300])
def test_exact_case_bit_exact(M):
    """x in {-1, 0, 1} with at most 8 nonzeros per row and s = 2^-6: every
    partial sum is exact in f32 and y*64 is an integer of magnitude <= 120, so
    y is exact in bfloat16 and every correct accumulation order gives the
    same bits as the oracle's exact value."""
    r = np.random.default_rng(100 + M)
    K, N = 256, 264
    xv = np.zeros((M, K))
    for m in range(M):
        nz = r.choice(K, size=8, replace=False)
        xv[m, nz] = r.choice([-1.0, 1.0], size=8)
    x = (xv.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    qw = r.integers(0, 1 << 32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32)
    qz = r.integers(0, 1 << 32, size=(K // 128, N // 8), dtype=np.uint64).astype(np.uint32)
    s = np.full((K // 128, N), 2.0 ** -6, dtype=np.float16).view(np.uint16)
    p = wi.Problem(M, K, N, 128, x, qw, s, qz)
    ref = oracle.gemm(x, qw, s, qz)
    want = oracle.f64_to_bf16(ref)
    assert np.array_equal(oracle.bf16_to_f64(want), ref)  # exact in bf16
    d = Device(p)
    for path in ([SPLITK, CS, TC] if M <= 8 else [TC]):
        got = bf16_bits(d.run(path))
        assert np.array_equal(got, want), f"path {path}: {np.count_nonzero(got != want)} bits differ"


@pytest.mark.parametrize("path", [AUTO, TC, SPLITK, CS])
def test_empty_batch_launches_nothing(path):
    """M = 0 (an empty batch): an empty result, no kernel launched."""
    import int4_weight_only_gemm_gb300 as w
    d = Device(wi.generate_named("qkv", 1, 0))
    x0 = torch.empty((0, d.prob.K), dtype=torch.bfloat16, device="cuda")
    before = w.w4a16_launch_count()
    y = d.run(path, x=x0)
    torch.cuda.synchronize()
    assert tuple(y.shape) == (0, d.prob.N)
    assert w.w4a16_launch_count() == before


def test_zero_codes_give_zero():
    K, N, M = 512, 256, 4
    r = np.random.default_rng(1)
    x = wi.f32_to_bf16_bits(r.standard_normal((M, K)).astype(np.float32))
    qw = np.zeros((K // 8, N), np.uint32)
    qz = np.zeros((K // 128, N // 8), np.uint32)
    s = wi.f64_to_f16_bits(r.uniform(0.001, 0.02, (K // 128, N)))
    d = Device(wi.Problem(M, K, N, 128, x, qw, s, qz))
    for path in (SPLITK, CS, TC):
        y = d.run(path)
        assert torch.count_nonzero(y.float()).item() == 0


# ---- determinism, workspace reuse, streams ------------------------------------

@pytest.mark.parametrize("shape,M,path", [("o_proj", 1, SPLITK), ("down", 4, SPLITK), ("o_proj", 1, CS),
                                          ("down", 8, CS), ("o_proj", 16, TC), ("down", 16, TC),
                                          ("qkv", 2048, TC)])
def test_deterministic_and_workspace_reused(shape, M, path):
    p = wi.generate_named(shape, M, 9)
    d = Device(p)
    import int4_weight_only_gemm_gb300 as w
    ws = w.new_workspace(w.w4a16_workspace_bytes(M, p.N, p.K, path=path))
    y1 = d.run(path, workspace=ws)
    y2 = d.run(path, workspace=ws)
    y3 = d.run(path, workspace=ws)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16))
    # counters are back at zero after every call
    nz = ws.view(torch.int32)[:16384].abs().sum().item() if ws.numel() >= 65536 else 0
    assert nz == 0
    check_sampled(d, y3, 1500, seed=1, what=f"{shape} M={M} reuse")


def test_registered_workspace_and_default_signature():
    import ctypes
    import int4_weight_only_gemm_gb300 as w
    p = wi.generate_named("qkv", 1, 11)
    d = Device(p)
    lib = w.load_library()
    need = w.w4a16_workspace_bytes(1, p.N, p.K)
    y = torch.empty((1, p.N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    if need:
        w.w4a16_set_workspace(None)
        st = lib.w4a16_gemm(d.x.data_ptr(), d.qd.data_ptr(), d.scales.data_ptr(), d.qzeros.data_ptr(),
                            1, p.N, p.K, 128, y.data_ptr(), stream)
        assert st == w.W4A16_EWORKSPACE
    ws = w.new_workspace(need)
    w.w4a16_set_workspace(ws)
    try:
        st = lib.w4a16_gemm(d.x.data_ptr(), d.qd.data_ptr(), d.scales.data_ptr(), d.qzeros.data_ptr(),
                            1, p.N, p.K, 128, y.data_ptr(), stream)
        assert st == 0
        torch.cuda.synchronize()
        _full(p, y, "registered workspace")
        assert w.w4a16_last_device_status() == 0
    finally:
        w.w4a16_set_workspace(None)
    # too small an explicit workspace is refused before launch
    if need:
        small = w.new_workspace(need // 2)
        st = w.w4a16_gemm_raw(d.x.data_ptr(), d.qd.data_ptr(), d.scales.data_ptr(), d.qzeros.data_ptr(),
                              1, p.N, p.K, 128, y.data_ptr(), small.data_ptr(), need // 2)
        assert st == w.W4A16_EWORKSPACE


def test_side_stream():
    p = wi.generate_named("o_proj", 16, 12)
    d = Device(p)
    import int4_weight_only_gemm_gb300 as w
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        y = w.w4a16_gemm(d.x, d.qd, d.scales, d.qzeros, stream=s)
    s.synchronize()
    _full(p, y, "side stream")


def test_gpu_argument_errors():
    import int4_weight_only_gemm_gb300 as w
    p = wi.generate_named("tiny", 1, 0)
    d = Device(p)
    with pytest.raises(w.W4A16Error) as e:
        w.w4a16_gemm(d.x, d.qd, d.scales[:1].contiguous(), d.qzeros[:1].contiguous(), group=256)
    assert e.value.status == w.W4A16_EUNSUPPORTED
    with pytest.raises(w.W4A16Error) as e:
        w.w4a16_gemm(d.x.repeat(9, 1), d.qd, d.scales, d.qzeros, path=GEMV)  # M=9 beyond the GEMV
    assert e.value.status == w.W4A16_EUNSUPPORTED
    assert w.w4a16_last_device_status() == 0


def test_one_workspace_across_shapes_and_paths():
    """A single workspace serves any sequence of calls: split-K partial sums
    of one problem must never disturb the arrival counters of the next."""
    import int4_weight_only_gemm_gb300 as w
    seq = [("down", 16, TC), ("gate_up", 1, SPLITK), ("o_proj", 1, SPLITK), ("vocab", 1, SPLITK),
           ("qkv", 16, TC), ("gate_up", 4, SPLITK), ("down", 2, CS)]
    need = max(w.w4a16_workspace_bytes(M, *reversed(wi.shape_kn(s)), path=pth) for s, M, pth in seq)
    ws = w.new_workspace(need)
    for i, (shape, M, path) in enumerate(seq):
        p = wi.generate_named(shape, M, 20 + i)
        d = Device(p)
        y = d.run(path, workspace=ws)
        check_sampled(d, y, 2000, seed=i, what=f"shared workspace {shape} M={M}")


# ---- launch flags: programmatic dependent launch ------------------------------

@pytest.mark.parametrize("flags", [0, 1, 3])
@pytest.mark.parametrize("shape,M,path", [("qkv", 1, GEMV), ("down", 8, GEMV), ("qkv", 1, SPLITK),
                                          ("down", 8, SPLITK), ("o_proj", 16, TC), ("gate_up", 64, TC),
                                          ("down", 300, TC)])
def test_launch_flags_same_result(flags, shape, M, path):
    """Every flag combination gives the same bits (the flags change launch
    overlap only) and matches the oracle."""
    p = wi.generate_named(shape, M, 30)
    d = Device(p)
    base = d.run(path, flags=0)
    y = d.run(path, flags=flags)
    torch.cuda.synchronize()
    assert torch.equal(base.view(torch.int16), y.view(torch.int16))
    check_sampled(d, y, 1500, seed=2, what=f"flags={flags} {shape} M={M}")


@pytest.mark.parametrize("M,path", [(1, GEMV), (4, GEMV), (1, SPLITK), (2, CS), (16, TC), (256, TC)])
@pytest.mark.parametrize("flags", [1, 3])
def test_chained_layers_respect_order(M, path, flags):
    """Layer 2 reads layer 1's output as its x.  Launched back to back as
    programmatic dependents, layer 2 must still see the finished y1: y1's
    buffer starts as NaN, so reading it early would show."""
    import int4_weight_only_gemm_gb300 as w
    p1 = wi.generate(M, 1024, 2048, seed=41)
    p2 = wi.generate(M, 2048, 512, seed=42)
    d1, d2 = Device(p1), Device(p2)
    for _ in range(3):
        y1 = torch.full((M, 2048), float("nan"), dtype=torch.bfloat16, device="cuda")
        y2 = torch.full((M, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        d1.run(path, flags=flags, out=y1)
        d2.run(path, x=y1, flags=flags, out=y2)
        torch.cuda.synchronize()
        x2 = bf16_bits(y1)
        assert np.all(np.isfinite(oracle.bf16_to_f64(x2[:1])))
        ref = oracle.gemm(x2, p2.qweight, p2.scales, p2.qzeros)
        check_close(bf16_to_f64(y2), ref, f"chain M={M} flags={flags}")
    assert w.w4a16_last_device_status() == 0


def _dispatch_rows():
    """Rows of the generated dispatch table (int4_weight_only_gemm_gb300/csrc/dispatch_table.h)."""
    import re
    hdr = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "int4_weight_only_gemm_gb300",
                       "csrc", "dispatch_table.h")
    text = open(hdr).read()
    paths = {"W4A16_PATH_GEMV_SPLITK": SPLITK, "W4A16_PATH_GEMV_CS": CS, "W4A16_PATH_TC": TC}
    rows = [(int(c), int(m), paths[p], int(nt)) for c, m, p, nt in
            re.findall(r"\{(\d+), (\d+), (W4A16_PATH_\w+), (\d+)\}", text)]
    limits = [int(v) for v in re.search(r"kClassMaxWeights\[\] = \{([^}]*)\}", text).group(1)
              .replace("ll", "").split(",")]
    return rows, limits


def test_auto_path_follows_the_dispatch_table():
    """AUTO picks the generated table's kernel for every shape of the decoder
    and the vocabulary head, at M inside and between the measured points."""
    import int4_weight_only_gemm_gb300 as w
    rows, limits = _dispatch_rows()
    assert rows
    for shape in list(wi.LAYER) + ["vocab"]:
        K, N = wi.shape_kn(shape)
        cls = sum(K * N > v for v in limits)
        mine = [r for r in rows if r[0] == cls]
        for M in (1, 2, 3, 4, 5, 8, 9, 16, 20, 33, 64, 100, 128, 300, 2048, 8192, 9000):
            row = next((r for r in mine if M <= r[1]), mine[-1])
            want = row[2] if M <= 8 or row[2] == TC else TC
            assert w.w4a16_auto_path(M, N, K) == want, (shape, M, row)
