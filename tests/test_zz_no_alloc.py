"""The backward entry point that allocates nothing (invrope_postmix_bwd_noalloc).

It exists for callers that may not allocate device memory on their call path
and have no workspace to pass; the dM partials then live in the library's own
fixed scratch array. Its results must match the regular backward (which takes
a caller workspace) within the tolerances of the other parity tests, on two
calls in a row. Before them, a call on other inputs fills the shared array
with different partials, so a partial the checked calls failed to write would
show up; the checked calls must also give the bits of the regular backward,
since the same kernels run. This file is collected last so that a run
stopping at the first failure has already run every other test."""

import pytest
import torch

import partial_inverse_rope_gb300 as ir
from gpu_helpers import assert_bf16_close, assert_dm_close, ensure_built, f64, make_inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 8 << 20  # INVROPE_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module", autouse=True)
def built():
    ensure_built()
    yield
    assert ir.invrope_take_device_fault() == 0


def _prime_scratch():
    """Fill the shared scratch with partials of other inputs, over at least
    the bytes every checked call uses (152 thread blocks of 64 x 64 partials),
    so that a partial a checked call failed to write would show up."""
    sq, nh, nope, pe = 2048, 64, 448, 64
    O, dY, M = make_inputs(sq, nh, nope, pe, seed=99)
    dO = torch.empty_like(O)
    dM = torch.empty(nh, nh, dtype=torch.float32, device="cuda")
    ir.invrope_postmix_bwd_noalloc(dY, O, M, 0, nope, pe, dO, dM)
    torch.cuda.synchronize()


@pytest.mark.parametrize("sq,nh,nope,pe,pos0", [
    (16384, 64, 448, 64, 16384),   # the production shard
    (2053, 16, 448, 64, 0),
    (37, 3, 56, 8, 5),
    (300, 64, 480, 64, 9),         # pe block across a 64-channel boundary (general tiling)
])
def test_noalloc_matches_workspace_backward_twice(sq, nh, nope, pe, pos0):
    assert ir.invrope_postmix_bwd_workspace_bytes(sq, nh, nope, pe) <= SCRATCH_BYTES
    O, dY, M = make_inputs(sq, nh, nope, pe, seed=sq)
    dO_ref, dM_ref = ir.invrope_postmix_bwd(dY, O, M, pos0, nope, pe)
    ref_dO, ref_dM = f64(dO_ref), f64(dM_ref)
    _prime_scratch()
    for call in range(2):
        dO = torch.empty_like(O)
        dM = torch.empty(nh, nh, dtype=torch.float32, device="cuda")
        ir.invrope_postmix_bwd_noalloc(dY, O, M, pos0, nope, pe, dO, dM)
        torch.cuda.synchronize()
        assert_bf16_close(f64(dO), ref_dO, f"dO (call {call + 1})")
        assert_dm_close(f64(dM), ref_dM, f"dM (call {call + 1})")
        # the same kernels run with the same partial layout: the bits agree too
        assert torch.equal(dO, dO_ref), f"dO bits (call {call + 1})"
        assert torch.equal(dM, dM_ref), f"dM bits (call {call + 1})"


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # 128 heads: one 64 KiB partial per thread block, more than 8 MiB in total
    sq, nh, nope, pe = 64, 128, 448, 64
    assert ir.invrope_postmix_bwd_workspace_bytes(sq, nh, nope, pe) > SCRATCH_BYTES
    O, dY, M = make_inputs(sq, nh, nope, pe, seed=1)
    dO = torch.empty_like(O)
    dM = torch.empty(nh, nh, dtype=torch.float32, device="cuda")
    with pytest.raises(ir.InvropeError, match="WORKSPACE"):
        ir.invrope_postmix_bwd_noalloc(dY, O, M, 0, nope, pe, dO, dM)
