"""GPU parity of the fused gate/up projection with the SiLU-multiply epilogue
(w4a16_pack_gate_up + w4a16_gemm_gate_up_silu, through the C ABI) against the
CPU oracle: pack bit-exact, outputs within the GEMM tolerance, on both kernels,
whole and split-K tiles, ragged token tiles, the decoder's 2560 x 19456 shape.
"""
import numpy as np
import pytest
import torch

import oracle
import w4a16_inputs as wi
from tests.gpu_helpers import bf16_to_f64, check_close

pytestmark = pytest.mark.gpu

GEMV, TC, AUTO, SPLITK, CS = 1, 2, 0, 3, 4


class Fused:
    def __init__(self, M, K, H, seed):
        import int4_weight_only_gemm_gb300 as w
        self.w = w
        self.H = H
        self.prob = wi.generate(M, K, 2 * H, seed=seed)
        self.x, self.qw, self.scales, self.qzeros = w.to_device(self.prob)
        self.qd = w.w4a16_pack_gate_up(self.qw)

    def run(self, path=AUTO, flags=None):
        return self.w.w4a16_gemm_gate_up_silu(self.x, self.qd, self.scales, self.qzeros, path=path, flags=flags)

    def ref(self):
        p = self.prob
        return oracle.gemm_gate_up_silu(p.x, p.qweight, p.scales, p.qzeros, self.H)


@pytest.mark.parametrize("K,H", [(128, 64), (384, 192), (2560, 9728)])
def test_pack_gate_up_bit_exact(K, H):
    import int4_weight_only_gemm_gb300 as w
    p = wi.generate(1, K, 2 * H, seed=K + H)
    _, qw, _, _ = w.to_device(p)
    qd = w.w4a16_pack_gate_up(qw)
    want = oracle.device_layout_gate_up(p.qweight, H)
    got = qd.cpu().numpy().view(np.uint32).reshape(-1)
    assert np.array_equal(got, want), f"{np.count_nonzero(got != want)} words differ"
    back = w.w4a16_unpack_gate_up(qd)
    assert torch.equal(back, qw)


@pytest.mark.parametrize("M,path", [(1, GEMV), (1, TC), (3, GEMV), (3, TC), (8, GEMV), (16, TC), (33, TC),
                                    (100, TC), (300, TC), (1, CS), (2, CS), (8, CS), (1, SPLITK)])
@pytest.mark.parametrize("K,H", [(128, 64), (512, 192), (1024, 320)])
def test_gate_up_small_full(M, K, H, path):
    f = Fused(M, K, H, seed=M * 31 + K + H)
    check_close(bf16_to_f64(f.run(path)), f.ref(), f"gate_up M={M} K={K} H={H} path={path}")


@pytest.mark.parametrize("M,path", [(1, GEMV), (2, GEMV), (1, TC), (16, TC), (64, TC), (1, CS), (2, SPLITK)])
def test_gate_up_split_k_tiles(M, path):
    # 20 column tiles, fewer than the SMs: every tile is cut into K pieces
    f = Fused(M, 9728, 1280, seed=70 + M)
    check_close(bf16_to_f64(f.run(path)), f.ref(), f"gate_up split M={M} path={path}")


@pytest.mark.parametrize("M,path", [(1, AUTO), (16, AUTO), (1, SPLITK), (2, CS)])
def test_gate_up_layer_shape_full(M, path):
    K, N = wi.shape_kn("gate_up")
    f = Fused(M, K, N // 2, seed=M)
    check_close(bf16_to_f64(f.run(path)), f.ref(), f"gate_up layer M={M} path={path}")


# The decoder's shape at M=2048 is checked in full in test_gemm.py, against the
# same oracle product as the plain GEMM of those weights.


def test_gate_up_flags_agree():
    import int4_weight_only_gemm_gb300 as w
    f = Fused(2, 2560, 640, seed=5)
    for path in (SPLITK, CS):
        base = f.run(path, flags=0)
        for flags in (w.FLAG_PDL, w.FLAG_PDL | w.FLAG_STATIC_WEIGHTS):
            assert torch.equal(f.run(path, flags=flags), base)


def test_gate_up_argument_errors():
    import int4_weight_only_gemm_gb300 as w
    lib = w.load_library()
    f = Fused(1, 128, 64, seed=1)
    y = torch.empty((1, 64), dtype=torch.bfloat16, device="cuda")
    ws = w.new_workspace(w.w4a16_workspace_bytes(1, 128, 128), "cuda")
    args = lambda H: (0, w.FLAG_PDL, f.x.data_ptr(), f.qd.data_ptr(), f.scales.data_ptr(), f.qzeros.data_ptr(), 1,
                      H, 128, 128, y.data_ptr(), ws.data_ptr(), ws.numel(), 0)
    assert lib.w4a16_gemm_gate_up_silu(*args(64)) == w.W4A16_OK
    assert lib.w4a16_gemm_gate_up_silu(*args(32)) == w.W4A16_EUNSUPPORTED  # H % 64 != 0
    assert lib.w4a16_gemm_gate_up_silu(*args(0)) == w.W4A16_EINVAL
    qw = torch.zeros((16, 96), dtype=torch.int32, device="cuda")
    assert lib.w4a16_pack_gate_up(qw.data_ptr(), torch.empty_like(qw).data_ptr(), 128, 48, 0) == w.W4A16_EUNSUPPORTED
    torch.cuda.synchronize()
