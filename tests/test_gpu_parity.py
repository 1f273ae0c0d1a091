"""CUDA path (through the C-ABI binding) against the fp64 oracle, element by
element, on seeded inputs; plus bitwise repeatability, exact special cases and
the launch-time error paths. Needs a GB300 (sm_103a)."""

import numpy as np
import pytest
import torch

import oracle
import partial_inverse_rope_gb300 as ir
from partial_inverse_rope_gb300 import binding
from gpu_helpers import assert_bf16_close, assert_dm_close, compare_all_rows, ensure_built, f64, make_inputs
from partial_inverse_rope_gb300 import inputs as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    ensure_built()
    yield
    assert ir.invrope_take_device_fault() == 0, "a kernel wait ran out during the tests"


def _full_check(sq, nh, nope, pe, pos0=0, theta=1e4, seed=0):
    O, dY, M = make_inputs(sq, nh, nope, pe, seed)
    Y = ir.invrope_postmix_fwd(O, M, pos0, nope, pe, theta)
    dO, dM = ir.invrope_postmix_bwd(dY, O, M, pos0, nope, pe, theta)
    torch.cuda.synchronize()
    pos = np.arange(pos0, pos0 + sq, dtype=np.int64)
    O64, dY64, M64 = f64(O), f64(dY), f64(M)
    Y_ref = oracle.postmix_fwd(O64, M64, pos, nope, pe, theta)
    dO_ref, dM_ref = oracle.postmix_bwd(dY64, O64, M64, pos, nope, pe, theta)
    assert_bf16_close(f64(Y), Y_ref, "Y")
    assert_bf16_close(f64(dO), dO_ref, "dO")
    assert_dm_close(f64(dM), dM_ref)


# ------------------------------------------------------------------ first launches
def test_0_one_row_one_column_remap():
    idx = torch.tensor([[3]], dtype=torch.int32, device="cuda")
    out = ir.kv_idx_local_to_global(idx, 1, 10)
    assert out.cpu().tolist() == [[3]]


def test_0_one_row_postmix():
    _full_check(1, 4, 48, 16)


# ------------------------------------------------------------------ postmix shapes
SHAPES = [
    # sq, nh, nope, pe, pos0, theta
    (1, 1, 6, 2, 0, 1e4),             # smallest: one head, one pair, d = 8
    (128, 4, 48, 16, 0, 1e4),         # the tiny config's shape
    (37, 3, 56, 8, 5, 1e4),           # nh=3, pe/2 = 4 (scalar rotation path), ragged rows
    (100, 5, 448, 64, 0, 1e4),        # 25 positions per tile, R = 125 rows
    (41, 7, 448, 64, 3, 1e4),         # R = 126 rows
    (65, 1, 448, 64, 0, 1e4),         # one head: 32 positions per tile
    (1000, 2, 112, 16, 7, 1e4),       # d = 128
    (300, 16, 136, 32, 11, 1e4),      # d = 168: ragged 64-channel chunk, pe inside it
    (257, 64, 0, 64, 0, 1e4),         # nope = 0: every channel rotated
    (1, 64, 448, 64, 0, 1e4),         # nh = 64 stacked backward mix, one position of two
    (301, 64, 480, 32, 9, 1e4),       # nh = 64 with pe < 64: block-diagonal backward mix
    (130, 64, 448, 64, 2**31 + 12345, 1e4),  # positions beyond 2^31 (exact angle reduction)
    (33, 128, 448, 64, 0, 5e5),       # 128 heads, another rotary base
    (70, 100, 448, 64, 3, 1e4),       # nh = 100: 128-channel backward tiles of R = 100 rows
    (40, 128, 64, 64, 0, 1e4),        # d = 128: one 128-channel tile per row tile, every tile has pe
    (50, 96, 480, 32, 5, 1e4),        # 128-channel backward tiles, pe = 32 in the last 64-channel chunk
    (2053, 16, 448, 64, 0, 1e4),      # mid-like, ragged
    (777, 32, 448, 64, 1, 1e4),       # nh = 32: 4 positions per tile
    (515, 48, 448, 64, 2, 1e4),       # nh = 48: 2 positions, R = 96, block-diagonal backward mix
    (200, 24, 100, 28, 4, 1e4),       # pe/2 = 14 (scalar rotation path), pe block inside chunk 1
    (90, 128, 510, 2, 6, 1e4),        # 128 heads, the smallest pe (one pair) at the end of d = 512
    # the pe block across a 64-channel boundary, or wider than 64: pair blocks of
    # the general tiling (nope tiles clipped at channel nope, pairs stored directly)
    (300, 64, 480, 64, 9, 1e4),       # 448 + 64 shifted by 32 channels
    (100, 16, 40, 32, 3, 1e4),
    (77, 128, 96, 64, 5, 1e4),        # 128 heads: one position per tile
    (50, 3, 120, 16, 2, 1e4),
    (64, 8, 384, 128, 7, 1e4),        # pe = 128: two pair blocks
    (45, 5, 0, 512, 11, 1e4),         # every channel rotated, 8 pair blocks
    (70, 12, 62, 10, 3, 1e4),         # nope % 8 != 0 and pe / 2 odd: unaligned pairs
    (33, 6, 60, 100, 4, 1e4),         # 50 pairs from channel 60: unaligned, two pair blocks
    (20, 64, 2, 254, 1, 1e4),         # 127 pairs, 64 heads
    (40, 7, 220, 76, 2**31 + 5, 5e5), # unaligned pairs, positions beyond 2^31, another base
    (131, 100, 448, 72, 8, 1e4),      # 36 pairs (a 4-pair second block), 100 heads
    # 128-channel backward tiles with many positions per tile (tensors of 1 MiB or more)
    (3000, 2, 448, 64, 1, 1e4),       # 64 positions per tile, R = 128
    (5000, 1, 448, 64, 0, 1e4),       # 64 positions per tile, R = 64
    (2100, 3, 160, 32, 3, 1e4),       # 42 positions (R = 126), pe tile every second tile
]


@pytest.mark.parametrize("sq,nh,nope,pe,pos0,theta", SHAPES)
def test_postmix_parity(sq, nh, nope, pe, pos0, theta):
    _full_check(sq, nh, nope, pe, pos0, theta, seed=sq + nh)


def test_tiny_config():
    c = W.TINY
    _full_check(c.sq, c.nh, c.nope, c.pe, c.pos0, c.theta, seed=c.seed)


def test_mid_config():
    c = W.MID
    _full_check(c.sq, c.nh, c.nope, c.pe, c.pos0, c.theta, seed=c.seed)


def test_sweep_nh3_config():
    c = W.SWEEP_NH3
    _full_check(c.sq, c.nh, c.nope, c.pe, c.pos0, c.theta, seed=c.seed)


def _large_check(c):
    """Full-size run: every row of Y and dO against the oracle (in blocks of
    rows, to bound host memory), dM against the full oracle sum."""
    O, dY, M = W.postmix_inputs(c, device="cuda")
    Y = ir.invrope_postmix_fwd(O, M, c.pos0, c.nope, c.pe, c.theta)
    dO, dM = ir.invrope_postmix_bwd(dY, O, M, c.pos0, c.nope, c.pe, c.theta)
    torch.cuda.synchronize()
    all_pos = np.arange(c.pos0, c.pos0 + c.sq, dtype=np.int64)
    compare_all_rows(O, dY, M, Y, dO, all_pos, c.nope, c.pe, c.theta)
    O32 = O.cpu().to(torch.float32).numpy()
    dY32 = dY.cpu().to(torch.float32).numpy()
    dM_ref = oracle.postmix_bwd_dM(dY32, O32, all_pos, c.nope, c.pe, c.theta)
    return assert_dm_close(f64(dM), dM_ref)


def test_production_shard_full_size():
    _large_check(W.PROD)


def test_sweep_nh128_full_size():
    _large_check(W.SWEEP_NH128)


def test_many_rows_small_channels():
    """2^27 + rows of the [sq*nh, d] view: large row coordinates, every row compared."""
    sq, nh, nope, pe = 2_097_159, 64, 0, 8
    O, dY, M = make_inputs(sq, nh, nope, pe, seed=5)
    Y = ir.invrope_postmix_fwd(O, M, 9, nope, pe, 1e4)
    dO, _ = ir.invrope_postmix_bwd(dY, O, M, 9, nope, pe, 1e4)
    torch.cuda.synchronize()
    compare_all_rows(O, dY, M, Y, dO, np.arange(9, 9 + sq, dtype=np.int64), nope, pe, 1e4,
                     block=65536)


# ------------------------------------------------------------------ exact special cases
def test_identity_mix_at_position_zero_is_exact():
    O, dY, _ = make_inputs(1, 64, 448, 64, seed=3)
    I = torch.eye(64, device="cuda")
    Y = ir.invrope_postmix_fwd(O, I, 0, 448, 64)
    dO, _ = ir.invrope_postmix_bwd(dY, O, I, 0, 448, 64)
    assert torch.equal(Y, O)
    assert torch.equal(dO, dY)


def test_permutation_mix_at_position_zero_is_exact():
    nh = 16
    O, _, _ = make_inputs(1, nh, 448, 64, seed=4)
    perm = torch.randperm(nh, generator=torch.Generator().manual_seed(0))
    P = torch.zeros(nh, nh)
    P[torch.arange(nh), perm] = 1.0
    Y = ir.invrope_postmix_fwd(O, P.cuda(), 0, 448, 64)
    assert torch.equal(Y[0], O[0, perm.cuda()])


def test_identity_mix_is_pure_inverse_rope():
    sq, nh, nope, pe = 300, 8, 448, 64
    O, _, _ = make_inputs(sq, nh, nope, pe, seed=6)
    Y = ir.invrope_postmix_fwd(O, torch.eye(nh, device="cuda"), 100, nope, pe)
    pos = np.arange(100, 100 + sq, dtype=np.int64)
    assert_bf16_close(f64(Y), oracle.invrope(f64(O), pos, nope, pe, 1e4), "Y = invrope(O)")
    assert torch.equal(Y[..., :nope], O[..., :nope])


def test_bitwise_repeatable():
    c = W.MID
    O, dY, M = W.postmix_inputs(c, device="cuda")
    outs = []
    for _ in range(3):
        Y = ir.invrope_postmix_fwd(O, M, c.pos0, c.nope, c.pe, c.theta)
        dO, dM = ir.invrope_postmix_bwd(dY, O, M, c.pos0, c.nope, c.pe, c.theta)
        outs.append((Y.clone(), dO.clone(), dM.clone()))
    for Y, dO, dM in outs[1:]:
        assert torch.equal(Y, outs[0][0])
        assert torch.equal(dO, outs[0][1])
        assert torch.equal(dM, outs[0][2])


@pytest.mark.parametrize("sq,nh,nope,pe", [(1024, 128, 448, 64), (4096, 2, 160, 32)])
def test_wide_backward_bitwise_repeatable(sq, nh, nope, pe):
    """The 128-channel backward issues a pe tile's dM chain before the next
    tile's data is waited for: the issue order is still fixed by the tile
    sequence, so repeated calls give the same bits."""
    O, dY, M = make_inputs(sq, nh, nope, pe, seed=21)
    dO0, dM0 = ir.invrope_postmix_bwd(dY, O, M, 5, nope, pe)
    for _ in range(5):
        dO, dM = ir.invrope_postmix_bwd(dY, O, M, 5, nope, pe)
        assert torch.equal(dO, dO0)
        assert torch.equal(dM, dM0)
    torch.cuda.synchronize()
    assert ir.invrope_take_device_fault() == 0


@pytest.mark.parametrize("nh,nope,pe", [(64, 0, 64), (16, 0, 32), (64, 8, 56), (16, 0, 128), (32, 4, 60)])
def test_every_tile_a_pe_tile_repeated(nh, nope, pe):
    """One channel tile, so every backward tile carries pe channels and the
    hand-offs to the transform warps come back to back; many calls in a row
    must all finish (no wait runs out) with bitwise identical results."""
    sq = 8192
    O, dY, M = make_inputs(sq, nh, nope, pe, seed=12)
    dO0, dM0 = ir.invrope_postmix_bwd(dY, O, M, 3, nope, pe)
    for _ in range(12):
        dO, dM = ir.invrope_postmix_bwd(dY, O, M, 3, nope, pe)
        assert torch.equal(dO, dO0)
        assert torch.equal(dM, dM0)
    torch.cuda.synchronize()
    assert ir.invrope_take_device_fault() == 0
    dO_ref, dM_ref = oracle.postmix_bwd(f64(dY), f64(O), f64(M), np.arange(3, 3 + sq, dtype=np.int64), nope, pe,
                                        1e4)
    assert_bf16_close(f64(dO0), dO_ref, "dO")
    assert_dm_close(f64(dM0), dM_ref)


@pytest.mark.parametrize("sq,nh,nope,pe,pos0", [
    (4096, 64, 448, 64, 16384),   # the stacked mix: static shares plus tail blocks
    (8192, 64, 480, 64, 7),       # general tiling, 128-channel tiles, two positions per tile
])
def test_backward_tail_blocks_exact_and_repeatable(sq, nh, nope, pe, pos0):
    """Shapes with enough tiles per CTA run a static share per CTA and then
    claim tail blocks dynamically: which CTA runs which block changes from call
    to call, dO and dM must not (every block has its own dM partial slot)."""
    O, dY, M = make_inputs(sq, nh, nope, pe, seed=sq + 5)
    runs = [ir.invrope_postmix_bwd(dY, O, M, pos0, nope, pe) for _ in range(5)]
    torch.cuda.synchronize()
    for dO, dM in runs[1:]:
        assert torch.equal(dO, runs[0][0])
        assert torch.equal(dM, runs[0][1])
    assert ir.invrope_take_device_fault() == 0
    positions = np.arange(pos0, pos0 + sq, dtype=np.int64)
    Y = ir.invrope_postmix_fwd(O, M, pos0, nope, pe)
    compare_all_rows(O, dY, M, Y, runs[0][0], positions, nope, pe, 1e4)
    dM_ref = oracle.postmix_bwd_dM(f64(dY), f64(O), positions, nope, pe, 1e4)
    assert_dm_close(f64(runs[0][1]), dM_ref)


def test_bwd_with_no_rows_zeroes_dM():
    O = torch.empty(0, 4, 64, dtype=torch.bfloat16, device="cuda")
    M = torch.eye(4, device="cuda")
    dM = torch.full((4, 4), 7.0, device="cuda")
    _, dM = ir.invrope_postmix_bwd(O, O, M, 0, 48, 16, dM=dM)
    assert torch.count_nonzero(dM).item() == 0


def test_dM_is_overwritten_not_accumulated():
    O, dY, M = make_inputs(64, 4, 48, 16, seed=8)
    _, a = ir.invrope_postmix_bwd(dY, O, M, 0, 48, 16)
    b = torch.full_like(a, 1e6)
    ir.invrope_postmix_bwd(dY, O, M, 0, 48, 16, dM=b)
    assert torch.equal(a, b)


# ------------------------------------------------------------------ launch-time errors
def test_workspace_too_small_is_rejected():
    O, dY, M = make_inputs(64, 4, 48, 16, seed=9)
    need = ir.invrope_postmix_bwd_workspace_bytes(64, 4, 48, 16)
    assert need > 0
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ir.InvropeError, match="WORKSPACE"):
        ir.invrope_postmix_bwd(dY, O, M, 0, 48, 16, workspace=ws)


def test_overlapping_output_is_rejected():
    O, _, M = make_inputs(64, 4, 48, 16, seed=10)
    with pytest.raises(ir.InvropeError, match="INVALID_ARG"):
        ir.invrope_postmix_fwd(O, M, 0, 48, 16, Y=O)


# ------------------------------------------------------------------ KV index remap
def _remap_check(idx_cpu, sq, skv, inplace=False):
    idx = idx_cpu.cuda()
    want = oracle.kv_idx_local_to_global(idx_cpu.numpy(), sq, skv)
    if inplace:
        out = ir.kv_idx_local_to_global(idx, sq, skv, out=idx)
    else:
        out = ir.kv_idx_local_to_global(idx, sq, skv)
    assert np.array_equal(out.cpu().numpy(), want)


@pytest.mark.parametrize("b,sq,topk,skv", [
    (1, 1, 1, 5),
    (3, 5, 7, 1000),        # topk % 4 != 0: scalar path, small batches
    (4, 3, 8, 100),         # vector path, batches shorter than a chunk
    (2, 1024, 640, 16384),  # vector path, one boundary per chunk
    (3, 333, 2176, 4096),
    (5, 17, 3, 2**28),      # large offsets
])
def test_remap_parity(b, sq, topk, skv):
    g = torch.Generator().manual_seed(b * 1000 + topk)
    idx = torch.randint(0, skv, (b * sq, topk), generator=g, dtype=torch.int32)
    pad = torch.rand(b * sq, topk, generator=g) < 0.1
    idx[pad] = -1
    idx[0, 0] = -7  # any negative value is padding
    _remap_check(idx, sq, skv)


def test_remap_in_place():
    g = torch.Generator().manual_seed(1)
    idx = torch.randint(-1, 500, (4 * 64, 128), generator=g, dtype=torch.int32)
    _remap_check(idx, 64, 500, inplace=True)


def test_remap_unaligned_view():
    g = torch.Generator().manual_seed(2)
    base = torch.randint(-1, 50, (4 * 10 * 9 + 1,), generator=g, dtype=torch.int32).cuda()
    idx = base[1:].view(40, 9)  # 4-byte aligned, not 16-byte aligned
    want = oracle.kv_idx_local_to_global(idx.cpu().numpy(), 10, 50)
    assert np.array_equal(ir.kv_idx_local_to_global(idx, 10, 50).cpu().numpy(), want)


def test_remap_int32_limit():
    idx = torch.tensor([[0, 2**30 - 1, -1], [2**30 - 1, 0, -1]], dtype=torch.int32)
    _remap_check(idx, 1, 2**30)


def test_remap_config_full_size():
    c = W.REMAP
    idx = W.kv_index_table(c, device="cuda")
    out = ir.kv_idx_local_to_global(idx, c.sq, c.seqlen_kv)
    want = oracle.kv_idx_local_to_global(idx.cpu().numpy(), c.sq, c.seqlen_kv)
    assert np.array_equal(out.cpu().numpy(), want)
    out2 = ir.kv_idx_local_to_global(idx, c.sq, c.seqlen_kv)
    assert torch.equal(out, out2)


# ------------------------------------------------------------------ bounded waits
def test_watchdog_gives_up_and_context_stays_usable():
    """A wait that nothing completes must run out, record its code and return;
    the context keeps working afterwards."""
    code = ir.invrope_watchdog_selftest(50000)
    assert code == binding.INVROPE_WATCHDOG_SELFTEST_CODE
    _full_check(64, 4, 48, 16, seed=11)
    assert ir.invrope_take_device_fault() == 0
