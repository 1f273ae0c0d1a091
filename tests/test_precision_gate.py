"""The fp32-rotation gate of ``precision_gate.py`` on emulated kernels (CPU).

The gate must pass a kernel that mixes with M as bf16 hi + lo in fp32,
rotates the fp32 result and rounds once, and must reject kernels that touch a
bf16-rounded value anywhere in the rotation: the mixed result rounded before
the rotation, bf16 sine / cosine, bf16 products, or the inputs rotated and
rounded to bf16 before the mix (the unfused route's rotated copy). The
emulations run numpy float32 arithmetic; the exact values come from the fp64
oracle.
"""

import numpy as np
import pytest
import torch

import oracle
from precision_gate import pair_scale, rne_bf16, rotation_gate, ulp_bf16

SQ, NH, NOPE, PE, POS0, THETA = 96, 16, 448, 64, 16384, 1e4


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).to(
        torch.float32).numpy()


def _inputs():
    g = torch.Generator().manual_seed(3)
    O = torch.randn(SQ, NH, NOPE + PE, generator=g).to(torch.bfloat16).to(torch.float64).numpy()
    M = (torch.eye(NH) + 0.02 * torch.randn(NH, NH, generator=g)).numpy().astype(np.float64)
    return O, M


def _emulate(O, M, mode):
    """Forward Y on the pe channels, emulated in float32 / bf16 as `mode` says."""
    pos = np.arange(POS0, POS0 + SQ)
    h = PE // 2
    Mhi = _bf16(M)
    Mlo = _bf16(M.astype(np.float32) - Mhi)
    O32 = O.astype(np.float32)
    a = pos[:, None].astype(np.float64) * oracle.inv_freq(PE, THETA)[None, :]
    c = np.cos(a).astype(np.float32)[:, None, :]
    sn = np.sin(a).astype(np.float32)[:, None, :]
    if mode == "bf16_sincos":
        c, sn = _bf16(c), _bf16(sn)
    if mode == "rotate_inputs_then_mix":
        x1, x2 = O32[:, :, NOPE:NOPE + h], O32[:, :, NOPE + h:]
        X = np.concatenate([_bf16(x1 * c + x2 * sn), _bf16(x2 * c - x1 * sn)], axis=2)
        Z = np.matmul(Mhi[None], X) + np.matmul(Mlo[None], X)
        return _bf16(Z)
    Z = (np.matmul(Mhi[None], O32) + np.matmul(Mlo[None], O32))[:, :, NOPE:].astype(np.float32)
    if mode == "round_mix_first":
        Z = _bf16(Z)
    z1, z2 = Z[:, :, :h], Z[:, :, h:]
    if mode == "bf16_products":
        y1 = _bf16(z1 * c) + _bf16(z2 * sn)
        y2 = _bf16(z2 * c) - _bf16(z1 * sn)
    else:
        y1 = z1 * c + z2 * sn
        y2 = z2 * c - z1 * sn
    return _bf16(np.concatenate([y1, y2], axis=2))


def _exact(O, M):
    pos = np.arange(POS0, POS0 + SQ)
    return oracle.postmix_fwd(O, M, pos, NOPE, PE, THETA)[:, :, NOPE:]


def test_rne_bf16_matches_known_values():
    assert rne_bf16(1.0 + 2.0 ** -8) == 1.0            # tie -> even
    assert rne_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert rne_bf16(-3.0 - 2.0 ** -7) == -3.0 - 2.0 ** -6 or rne_bf16(-3.0 - 2.0 ** -7) == -3.0
    assert ulp_bf16(1.0) == 2.0 ** -7 and ulp_bf16(0.75) == 2.0 ** -8
    x = np.random.default_rng(0).standard_normal(10000)
    # agrees with torch's fp32 -> bf16 nearest-even rounding where fp32 is exact
    x32 = x.astype(np.float32).astype(np.float64)
    assert np.array_equal(rne_bf16(x32), _bf16(x32).astype(np.float64))


def test_fp32_rotation_rounded_once_passes():
    O, M = _inputs()
    got = _emulate(O, M, "fp32")
    bad, ulps = rotation_gate(got, _exact(O, M), pair_scale(O, np.abs(M).T, NOPE, PE))
    assert not bad.any(), f"{bad.sum()} elements outside the gate, max {ulps.max():.3f} ulp"
    assert np.mean(got == rne_bf16(_exact(O, M))) > 0.99


@pytest.mark.parametrize("mode", ["round_mix_first", "bf16_sincos", "bf16_products", "rotate_inputs_then_mix"])
def test_any_bf16_step_in_the_rotation_fails(mode):
    O, M = _inputs()
    got = _emulate(O, M, mode)
    bad, _ = rotation_gate(got, _exact(O, M), pair_scale(O, np.abs(M).T, NOPE, PE))
    assert bad.mean() > 0.01, f"{mode}: only {bad.mean():.4%} outside the gate"
