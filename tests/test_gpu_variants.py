"""The grouped head mix, per-row positions and the int64 KV remap: CUDA path
(through the C-ABI binding) against the fp64 oracle on seeded inputs, plus the
exact equalities with the plain entry points. Needs a GB300 (sm_103a)."""

import numpy as np
import pytest
import torch

import oracle
import partial_inverse_rope_gb300 as ir
from gpu_helpers import assert_bf16_close, assert_dm_close, compare_all_rows, ensure_built, f64
from partial_inverse_rope_gb300 import inputs as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    ensure_built()
    yield
    assert ir.invrope_take_device_fault() == 0, "a kernel wait ran out during the tests"


def _inputs(sq, nh, d, seed):
    return W.normal_bf16((sq, nh, d), seed, "cuda"), W.normal_bf16((sq, nh, d), seed + 1, "cuda")


# ------------------------------------------------------------------ grouped head mix
@pytest.mark.parametrize("sq,nh,gs,nope,pe", [
    (300, 64, 8, 448, 64),    # nh = 64: the stacked backward mix, 8 groups
    (257, 16, 4, 448, 64),
    (101, 6, 3, 56, 8),       # scalar rotation path, ragged rows
    (64, 12, 1, 48, 16),      # gs = 1: each head scaled by its own factor
    (33, 128, 32, 448, 64),
    (100, 16, 4, 40, 32),     # pe block across a 64-channel boundary (general tiling)
    (60, 64, 16, 480, 64),
])
def test_grouped_parity(sq, nh, gs, nope, pe):
    O, dY = _inputs(sq, nh, nope + pe, seed=sq + gs)
    Mg = W.postmix_Mg(nh // gs, gs, seed=7 + gs, device="cuda")
    Y = ir.invrope_postmix_fwd_ex(O, Mg, nope, pe, pos0=3, group_size=gs)
    dO, dMg = ir.invrope_postmix_bwd_ex(dY, O, Mg, nope, pe, pos0=3, group_size=gs)
    torch.cuda.synchronize()
    pos = np.arange(3, 3 + sq, dtype=np.int64)
    Y_ref = oracle.postmix_fwd_grouped(f64(O), f64(Mg), pos, nope, pe, 1e4)
    dO_ref, dM_ref = oracle.postmix_bwd_grouped(f64(dY), f64(O), f64(Mg), pos, nope, pe, 1e4)
    assert_bf16_close(f64(Y), Y_ref, "grouped Y")
    assert_bf16_close(f64(dO), dO_ref, "grouped dO")
    assert_dm_close(f64(dMg), dM_ref, "grouped dM")


def _block_diag(Mg):
    ng, gs, _ = Mg.shape
    M = torch.zeros(ng * gs, ng * gs, device=Mg.device)
    for k in range(ng):
        M[k * gs:(k + 1) * gs, k * gs:(k + 1) * gs] = Mg[k]
    return M


@pytest.mark.parametrize("nh,gs", [(64, 16), (8, 2)])
def test_grouped_equals_ungrouped_block_diagonal_bitwise(nh, gs):
    sq, nope, pe = 130, 448, 64
    O, dY = _inputs(sq, nh, nope + pe, seed=40 + nh)
    Mg = W.postmix_Mg(nh // gs, gs, seed=41, device="cuda")
    M = _block_diag(Mg)
    Yg = ir.invrope_postmix_fwd_ex(O, Mg, nope, pe, pos0=9, group_size=gs)
    dOg, dMg = ir.invrope_postmix_bwd_ex(dY, O, Mg, nope, pe, pos0=9, group_size=gs)
    Y = ir.invrope_postmix_fwd(O, M, 9, nope, pe)
    dO, dM = ir.invrope_postmix_bwd(dY, O, M, 9, nope, pe)
    assert torch.equal(Yg, Y)
    assert torch.equal(dOg, dO)
    for k in range(nh // gs):
        sl = slice(k * gs, (k + 1) * gs)
        assert torch.equal(dMg[k], dM[sl, sl])


def test_one_group_equals_plain_entry_points_bitwise():
    sq, nh, nope, pe = 200, 64, 448, 64
    O, dY = _inputs(sq, nh, nope + pe, seed=50)
    M = W.postmix_M(nh, 51, "cuda")
    assert torch.equal(ir.invrope_postmix_fwd_ex(O, M[None], nope, pe, pos0=5, group_size=nh),
                       ir.invrope_postmix_fwd(O, M, 5, nope, pe))
    dOg, dMg = ir.invrope_postmix_bwd_ex(dY, O, M[None], nope, pe, pos0=5, group_size=nh)
    dO, dM = ir.invrope_postmix_bwd(dY, O, M, 5, nope, pe)
    assert torch.equal(dOg, dO) and torch.equal(dMg[0], dM)


# ------------------------------------------------------------------ per-row positions
@pytest.mark.parametrize("sq,nh,nope,pe,low,high,pos0", [
    (301, 64, 448, 64, 0, 65536, 0),            # a context-parallel shard's scattered positions
    (257, 8, 112, 16, -5000, 5000, 0),          # negative positions
    (99, 5, 56, 8, 2**31 - 4096, 2**31 - 1, 77),  # near the int32 end, plus an offset
    (65, 1, 448, 64, 0, 1 << 20, 3),            # one head, 32 positions per tile
    (150, 16, 100, 156, -3000, 3000, 5),        # general tiling: 78 pairs from channel 100
])
def test_positions_parity(sq, nh, nope, pe, low, high, pos0):
    O, dY = _inputs(sq, nh, nope + pe, seed=sq)
    M = W.postmix_M(nh, 60, "cuda")
    pos = W.random_positions(sq, 61, low, high, "cuda")
    Y = ir.invrope_postmix_fwd_ex(O, M, nope, pe, positions=pos, pos0=pos0)
    dO, dM = ir.invrope_postmix_bwd_ex(dY, O, M, nope, pe, positions=pos, pos0=pos0)
    torch.cuda.synchronize()
    p = pos0 + pos.cpu().numpy().astype(np.int64)
    assert_bf16_close(f64(Y), oracle.postmix_fwd(f64(O), f64(M), p, nope, pe, 1e4), "Y")
    dO_ref, dM_ref = oracle.postmix_bwd(f64(dY), f64(O), f64(M), p, nope, pe, 1e4)
    assert_bf16_close(f64(dO), dO_ref, "dO")
    assert_dm_close(f64(dM), dM_ref)


def test_contiguous_positions_array_equals_pos0_bitwise():
    sq, nh, nope, pe = 300, 64, 448, 64
    O, dY = _inputs(sq, nh, nope + pe, seed=70)
    M = W.postmix_M(nh, 71, "cuda")
    pos = torch.arange(sq, dtype=torch.int32, device="cuda")
    assert torch.equal(ir.invrope_postmix_fwd_ex(O, M, nope, pe, positions=pos, pos0=1000),
                       ir.invrope_postmix_fwd(O, M, 1000, nope, pe))
    a = ir.invrope_postmix_bwd_ex(dY, O, M, nope, pe, positions=pos, pos0=1000)
    b = ir.invrope_postmix_bwd(dY, O, M, 1000, nope, pe)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_folded_sequences_full_size():
    """The production shard's token axis holding 4 sequences of 4096 tokens
    (positions restart per sequence); every row of Y and dO, and dM."""
    c = W.PROD
    O, dY, M = W.postmix_inputs(c, device="cuda")
    p64 = oracle.positions_batched(4, c.sq // 4, 0)
    pos = torch.from_numpy(p64.astype(np.int32)).cuda()
    Y = ir.invrope_postmix_fwd_ex(O, M, c.nope, c.pe, positions=pos)
    dO, dM = ir.invrope_postmix_bwd_ex(dY, O, M, c.nope, c.pe, positions=pos)
    torch.cuda.synchronize()
    compare_all_rows(O, dY, M, Y, dO, p64, c.nope, c.pe, c.theta)
    dM_ref = oracle.postmix_bwd_dM(dY.cpu().float().numpy(), O.cpu().float().numpy(), p64, c.nope, c.pe,
                                   c.theta)
    assert_dm_close(f64(dM), dM_ref)


def test_grouped_with_positions_is_repeatable_bitwise():
    sq, nh, gs, nope, pe = 2048, 64, 16, 448, 64
    O, dY = _inputs(sq, nh, nope + pe, seed=80)
    Mg = W.postmix_Mg(nh // gs, gs, 81, "cuda")
    pos = W.random_positions(sq, 82, 0, 1 << 24, "cuda")
    runs = [ir.invrope_postmix_bwd_ex(dY, O, Mg, nope, pe, positions=pos, group_size=gs) for _ in range(3)]
    for dO, dM in runs[1:]:
        assert torch.equal(dO, runs[0][0]) and torch.equal(dM, runs[0][1])


# ------------------------------------------------------------------ int64 KV remap
@pytest.mark.parametrize("b,sq,topk,skv", [
    (1, 1, 1, 5),
    (3, 5, 7, 1000),              # odd topk: scalar path
    (4, 16, 640, 2**33),          # offsets past 2^31
    (2, 512, 2176, 16384),        # vector path, one boundary per chunk
    (3, 4, 2, 3 * 2**40),
])
def test_remap_i64_parity(b, sq, topk, skv):
    g = torch.Generator().manual_seed(b * 7 + topk)
    idx = torch.randint(0, skv, (b * sq, topk), generator=g, dtype=torch.int64)
    idx[torch.rand(b * sq, topk, generator=g) < 0.1] = -1
    idx[0, 0] = -123
    out = ir.kv_idx_local_to_global_i64(idx.cuda(), sq, skv)
    want = oracle.kv_idx_local_to_global_i64(idx.numpy(), sq, skv)
    assert np.array_equal(out.cpu().numpy(), want)


def test_remap_i64_in_place_and_wrap():
    idx = torch.tensor([[2**62, -1], [2**62, 5]], dtype=torch.int64, device="cuda")
    ir.kv_idx_local_to_global_i64(idx, 1, 2**62, out=idx)
    assert idx.cpu().tolist() == [[2**62, -1], [-2**63, 2**62 + 5]]


def test_remap_i64_matches_int32_in_range():
    c = W.REMAP
    idx = W.kv_index_table(c, device="cuda")[: 4 * 1024]
    a = ir.kv_idx_local_to_global(idx, 1024, c.seqlen_kv)
    b = ir.kv_idx_local_to_global_i64(idx.to(torch.int64), 1024, c.seqlen_kv)
    assert torch.equal(a.to(torch.int64), b)


# ------------------------------------------------------------------ M placement
def test_forward_with_misaligned_M_matches_bitwise():
    """An M that is only 4-byte aligned takes the forward's L2 path instead of
    the bulk copy into shared memory; both give the same bits."""
    sq, nh, nope, pe = 300, 64, 448, 64
    O, dY = _inputs(sq, nh, nope + pe, seed=90)
    M = W.postmix_M(nh, 91, "cuda")
    flat = torch.empty(nh * nh + 1, dtype=torch.float32, device="cuda")
    M_off = flat[1:].view(nh, nh)
    M_off.copy_(M)
    assert M_off.data_ptr() % 16 != 0
    a = ir.invrope_postmix_fwd(O, M, 7, nope, pe)
    b = ir.invrope_postmix_fwd(O, M_off, 7, nope, pe)
    assert torch.equal(a, b)
    da = ir.invrope_postmix_bwd(dY, O, M, 7, nope, pe)
    db = ir.invrope_postmix_bwd(dY, O, M_off, 7, nope, pe)
    assert torch.equal(da[0], db[0]) and torch.equal(da[1], db[1])
