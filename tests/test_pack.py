"""GPU pack/unpack against the oracle's rendering of the documented device
layout: bit-exact, including ragged column tiles."""
import numpy as np
import pytest
import torch

import oracle
import w4a16_inputs as wi

pytestmark = pytest.mark.gpu

SHAPES = [(128, 8), (128, 128), (256, 136), (384, 264), (2560, 4096), (9728, 2560), (2560, 151936)]


def _codes(K, N, seed):
    r = np.random.default_rng(seed)
    return r.integers(0, 1 << 32, size=(K // 8, N), dtype=np.uint64).astype(np.uint32)


@pytest.mark.parametrize("K,N", SHAPES)
def test_pack_matches_documented_layout(K, N):
    import int4_weight_only_gemm_gb300 as w
    q = _codes(K, N, K + N)
    qt = torch.from_numpy(q.view(np.int32)).cuda()
    qd = w.w4a16_pack(qt)
    got = qd.cpu().numpy().view(np.uint32).ravel()
    want = oracle.device_layout(q)
    assert np.array_equal(got, want)
    back = w.w4a16_unpack(qd).cpu().numpy().view(np.uint32)
    assert np.array_equal(back, q)


@pytest.mark.parametrize("fill", [0, 0xFFFFFFFF, "ramp"])
def test_pack_structured(fill):
    import int4_weight_only_gemm_gb300 as w
    K, N = 256, 264
    if fill == "ramp":
        codes = ((np.arange(K)[:, None] + np.arange(N)[None, :]) % 16).astype(np.uint8)
        q = oracle.pack_codes(codes)
    else:
        q = np.full((K // 8, N), fill, dtype=np.uint32)
    qd = w.w4a16_pack(torch.from_numpy(q.view(np.int32)).cuda())
    assert np.array_equal(qd.cpu().numpy().view(np.uint32).ravel(), oracle.device_layout(q))
    assert np.array_equal(w.w4a16_unpack(qd).cpu().numpy().view(np.uint32), q)


def test_pack_on_side_stream():
    import int4_weight_only_gemm_gb300 as w
    q = _codes(512, 384, 7)
    qt = torch.from_numpy(q.view(np.int32)).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        qd = w.w4a16_pack(qt, stream=s)
    s.synchronize()
    assert np.array_equal(qd.cpu().numpy().view(np.uint32).ravel(), oracle.device_layout(q))
