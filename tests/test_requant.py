"""Grid-preserving re-quantization on the GPU against the oracle, bit for bit:
code = clamp(round(w / s) + z, 0, 15), written in the device layout
("Quantize the Target, Quantize the Drafter", pith.science review,
"Assumptions & free parameters")."""
import numpy as np
import pytest
import torch

import oracle
import w4a16_inputs as wi

pytestmark = pytest.mark.gpu


def _gpu(w_bits, scales, qzeros):
    import int4_weight_only_gemm_gb300 as w
    wt = torch.from_numpy(w_bits.view(np.int16)).cuda().view(torch.bfloat16)
    st = torch.from_numpy(scales.view(np.int16)).cuda().view(torch.float16)
    zt = torch.from_numpy(qzeros.view(np.int32)).cuda()
    out = w.w4a16_requant_pack(wt, st, zt)
    torch.cuda.synchronize()
    return out


def _want_words(codes):
    return oracle.device_layout(oracle.pack_codes(codes))


@pytest.mark.parametrize("K,N", [(256, 128), (256, 136), (2560, 4096), (9728, 2560), (2560, 19456)])
def test_bit_exact_against_oracle(K, N):
    p = wi.generate(1, K, N, seed=21, shape_index=7)  # scales and zeros of the frozen grid
    w_bits = wi.random_weights(K, N, seed=21)
    got = _gpu(w_bits, p.scales, p.qzeros).cpu().numpy().view(np.uint32).reshape(-1)
    codes = oracle.requant_codes(w_bits, p.scales, p.qzeros)
    want = _want_words(codes)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} of {want.size} words differ, first at {bad[:5]}"
    # the codes span the range, clipping included
    assert codes.min() == 0 and codes.max() == 15


def test_round_trip_from_dequantized_codes():
    """w = bf16((q - z) s) re-quantizes to the original codes q."""
    import int4_weight_only_gemm_gb300 as w
    p = wi.generate(1, 2560, 4096, seed=22, shape_index=8)
    w_bits = oracle.f64_to_bf16(oracle.dequant(p.qweight, p.scales, p.qzeros))
    got = _gpu(w_bits, p.scales, p.qzeros)
    want = w.w4a16_pack(torch.from_numpy(p.qweight.view(np.int32)).cuda())
    torch.cuda.synchronize()
    assert torch.equal(got, want)


def test_ties_round_to_even():
    K, N = 256, 128
    s = np.full((K // 128, N), 2.0 ** -6)
    j = np.arange(K * N).reshape(K, N) % 40 - 20  # half-integers -19.5 .. 19.5, exact in bf16
    w = ((j + 0.5) * 2.0 ** -6).astype(np.float32)
    zeros = np.full((K // 128, N), 8, dtype=np.uint8)
    w_bits, s_bits, qz = wi.f32_to_bf16_bits(w), wi.f64_to_f16_bits(s), oracle.pack_zeros(zeros)
    codes = oracle.requant_codes(w_bits, s_bits, qz)
    got = _gpu(w_bits, s_bits, qz).cpu().numpy().view(np.uint32).reshape(-1)
    assert np.array_equal(got, _want_words(codes))
    assert codes[0, 20] == 8 and codes[0, 21] == 10  # 0.5 -> 0, 1.5 -> 2


def test_argument_errors():
    import int4_weight_only_gemm_gb300 as w
    lib = w.load_library()
    K, N = 256, 128
    wt = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    st = torch.ones((K // 128, N), dtype=torch.float16, device="cuda")
    zt = torch.zeros((K // 128, N // 8), dtype=torch.int32, device="cuda")
    out = torch.empty((K // 8, N), dtype=torch.int32, device="cuda")
    ok = lib.w4a16_requant_pack(wt.data_ptr(), st.data_ptr(), zt.data_ptr(), K, N, 128, out.data_ptr(), None)
    assert ok == w.W4A16_OK
    assert lib.w4a16_requant_pack(wt.data_ptr(), st.data_ptr(), zt.data_ptr(), K, N, 64, out.data_ptr(), None) \
        == w.W4A16_EUNSUPPORTED
    assert lib.w4a16_requant_pack(wt.data_ptr() + 2, st.data_ptr(), zt.data_ptr(), K, N, 128, out.data_ptr(), None) \
        == w.W4A16_EALIGN
    assert lib.w4a16_requant_pack(wt.data_ptr(), st.data_ptr(), zt.data_ptr(), K, N, 128, wt.data_ptr(), None) \
        == w.W4A16_EINVAL
    assert lib.w4a16_requant_pack(None, st.data_ptr(), zt.data_ptr(), K, N, 128, out.data_ptr(), None) \
        == w.W4A16_EINVAL
    assert lib.w4a16_requant_pack(wt.data_ptr(), st.data_ptr(), zt.data_ptr(), K, 100, 128, out.data_ptr(), None) \
        == w.W4A16_EINVAL
    torch.cuda.synchronize()
