"""The pins are strong enough: plausible mistakes planted in a CPU rendering
of the definition are each caught by at least one pin.

Every mutant below is a copy of the numpy rendering with one deliberate bug
(the kind a from-scratch oracle could plausibly contain).  Nothing here runs
on a GPU.
"""
import numpy as np
import pytest

from tests import oracle_pins


def _decode(x, qweight, scales, qzeros, group, *, nib_rev=False, zrev=False,
            gidx_mod=False, drop_zero=False, flip=False, s_transposed=False,
            s_bf16=False, z_along_k=False, group_shift=False, x_trunc_hi=False):
    qweight = np.asarray(qweight, dtype=np.uint32)
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    sh = 4 * np.arange(8, dtype=np.uint32)
    if nib_rev:
        sh = sh[::-1].copy()
    q = ((qweight[:, None, :] >> sh[None, :, None]) & 0xF).reshape(K, N).astype(np.float64)
    qz = np.asarray(qzeros, dtype=np.uint32)
    zsh = 4 * np.arange(8, dtype=np.uint32)
    if zrev:
        zsh = zsh[::-1].copy()
    z = ((qz[:, :, None] >> zsh[None, None, :]) & 0xF).reshape(qz.shape[0], N).astype(np.float64)
    if z_along_k:
        z = z[::-1].copy()
    sb = np.asarray(scales, dtype=np.uint16)
    if s_bf16:
        s = (sb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        s = sb.view(np.float16).astype(np.float64)
    if s_transposed:
        s = s.T.reshape(s.shape).copy() if s.shape[0] != s.shape[1] else s.T.copy()
    G = K // group
    k = np.arange(K)
    gidx = (k % G) if gidx_mod else (k // group)
    if group_shift:
        gidx = np.minimum((k + 1) // group, G - 1)
    zz = 0.0 if drop_zero else z[gidx]
    W = (zz - q) if flip else (q - zz)
    W = W * s[gidx]
    xb = np.asarray(x, dtype=np.uint16).astype(np.uint32)
    if x_trunc_hi:
        xb = xb & 0xFF80
    xv = (xb << 16).view(np.float32).astype(np.float64)
    return xv @ W


MUTANTS = {
    "nibble_order_reversed": dict(nib_rev=True),
    "zero_nibble_order_reversed": dict(zrev=True),
    "group_index_modulo": dict(gidx_mod=True),
    "zero_point_dropped": dict(drop_zero=True),
    "sign_flipped": dict(flip=True),
    "scales_transposed": dict(s_transposed=True),
    "scales_read_as_bf16": dict(s_bf16=True),
    "zero_groups_reversed": dict(z_along_k=True),
    "group_boundary_off_by_one": dict(group_shift=True),
    "x_low_bits_dropped": dict(x_trunc_hi=True),
}


def test_unmutated_rendering_passes_all_pins():
    impl = lambda *a: _decode(*a)  # noqa: E731
    for pin in oracle_pins.ALL_PINS:
        pin(impl)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    kw = MUTANTS[name]
    impl = lambda *a: _decode(*a, **kw)  # noqa: E731
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(impl)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
