"""``high_precision_rope``: the rotation runs in fp32 on unrounded values and
its result is rounded to bf16 once, in the forward and in the backward's dO.

PaddleFleet PR #1772 (Chinese description section 1) and PR #1843 (item 1)
name ``high_precision_rope=True`` among the settings the fused path hands
back to the unfused code, without defining it. Read here as "no bf16 rounding
inside the rotation"; the fused kernels are built that way in every mode, so
this test checks that reading against the fp64 oracle with the gate of
``precision_gate.py`` (0.5 ulp of the exact value plus 2^-14 of the pair's
fp32 term magnitude), which emulated bf16 rotations fail on 20-30 % of their
outputs (``test_precision_gate.py``). Production positions (16384 onwards), 64
heads. Needs a GB300 (sm_103a)."""

import numpy as np
import pytest
import torch

import oracle
import partial_inverse_rope_gb300 as ir
from gpu_helpers import ensure_built, f64
from partial_inverse_rope_gb300 import inputs as W
from precision_gate import pair_scale, rne_bf16, rotation_gate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    ensure_built()
    yield
    assert ir.invrope_take_device_fault() == 0


def _report(what, got, exact, scale):
    bad, ulps = rotation_gate(got, exact, scale)
    equal = float(np.mean(got == rne_bf16(exact)))
    print(f"{what}: {exact.size} pe outputs, {equal:.5%} equal to RNE(exact), max {ulps.max():.3f} ulp, "
          f"{int(bad.sum())} outside the gate")
    assert not bad.any(), f"{what}: {int(bad.sum())} outputs outside the fp32-rotation gate"
    assert equal > 0.99, f"{what}: only {equal:.4%} equal to the once-rounded exact value"


@pytest.mark.parametrize("sq,nh,nope,pe,identity", [
    (2048, 64, 448, 64, True),     # M = I: Y = invrope(O) exactly, dO = rope(dY)
    (2048, 64, 448, 64, False),    # M = I + 0.02 N(0,1)
    (1024, 64, 480, 64, True),     # general tiling (pe block across a 64-channel boundary)
    (1024, 16, 448, 64, False),    # the block-diagonal head mix
])
def test_rotation_is_fp32_and_rounded_once(sq, nh, nope, pe, identity):
    c = W.PostmixConfig("precision", sq=sq, nh=nh, nope=nope, pe=pe, pos0=16384)
    O, dY, M = W.postmix_inputs(c, device="cuda")
    if identity:
        M = torch.eye(nh, device="cuda")
    Y = ir.invrope_postmix_fwd(O, M, c.pos0, nope, pe, c.theta)
    dO, _ = ir.invrope_postmix_bwd(dY, O, M, c.pos0, nope, pe, c.theta)
    torch.cuda.synchronize()
    pos = np.arange(c.pos0, c.pos0 + sq, dtype=np.int64)
    O64, dY64, M64 = f64(O), f64(dY), f64(M)
    Y_ex = oracle.postmix_fwd(O64, M64, pos, nope, pe, c.theta)[:, :, nope:]
    dO_ex = oracle.postmix_bwd_dO(dY64, M64, pos, nope, pe, c.theta)[:, :, nope:]
    tag = f"{'M = I' if identity else 'M = I + 0.02 N'}, {nope} + {pe}, nh {nh}"
    _report(f"Y ({tag})", f64(Y)[:, :, nope:], Y_ex, pair_scale(O64, np.abs(M64).T, nope, pe))
    _report(f"dO ({tag})", f64(dO)[:, :, nope:], dO_ex, pair_scale(dY64, np.abs(M64), nope, pe))
