"""The C-ABI library without a GPU: it builds, loads, exports every symbol that
``include/invrope.h`` declares, and rejects bad arguments on the host before
touching CUDA. No call here reaches a kernel launch."""

import ctypes
import os
import re

import pytest
import torch

import partial_inverse_rope_gb300 as ir
from partial_inverse_rope_gb300 import binding
from partial_inverse_rope_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "invrope.h")

OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.lib_path()):
        build()
    return binding.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\(", text)
    skip = {"if", "defined", "sizeof"}
    return sorted({n for n in names if n not in skip and (n.startswith("invrope_") or n.startswith("kv_"))})


def test_header_declares_the_expected_entry_points():
    assert _declared_functions() == sorted([
        "invrope_last_cuda_error", "invrope_postmix_bwd", "invrope_postmix_bwd_workspace_bytes",
        "invrope_postmix_bwd_noalloc", "invrope_postmix_fwd", "invrope_status_string",
        "invrope_take_device_fault", "invrope_watchdog_selftest", "kv_idx_local_to_global",
        "invrope_postmix_fwd_ex", "invrope_postmix_bwd_ex", "kv_idx_local_to_global_i64",
        "invrope_debug_occupy_next_slot"])


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_binding_signatures_cover_the_header():
    assert set(_declared_functions()) <= set(binding._SIGNATURES)


def test_status_strings(lib):
    for code in range(6):
        s = lib.invrope_status_string(code).decode()
        assert s.startswith("INVROPE_"), s
    assert lib.invrope_status_string(99).decode() == "INVROPE_ERR_UNKNOWN"


FAKE = 0x10000  # never dereferenced: every call below is rejected on the host


@pytest.mark.parametrize("sq,nh,nope,pe,pos0,theta,want", [
    (8, 0, 448, 64, 0, 1e4, INVALID),        # no heads
    (8, 4, 448, 63, 0, 1e4, INVALID),        # odd pe
    (8, 4, 448, 0, 0, 1e4, INVALID),         # pe = 0
    (8, 4, 44, 16, 0, 1e4, INVALID),         # d not a multiple of 8
    (-1, 4, 48, 16, 0, 1e4, INVALID),        # negative rows
    (8, 4, 48, 16, -1, 1e4, INVALID),        # negative position
    (8, 4, 48, 16, 0, 0.0, INVALID),         # theta <= 0
    (8, 4, 48, 16, 0, float("inf"), INVALID),
    (8, 129, 448, 64, 0, 1e4, UNSUPPORTED),  # more than 128 heads
    (2**30, 4, 448, 64, 0, 1e4, UNSUPPORTED),  # sq * nh >= 2^31: beyond 32-bit row coordinates
])
def test_fwd_rejects_bad_shapes(lib, sq, nh, nope, pe, pos0, theta, want):
    st = lib.invrope_postmix_fwd(FAKE, FAKE, FAKE * 2, sq, nh, nope, pe, pos0, theta, None)
    assert st == want


@pytest.mark.parametrize("nh,nope,pe", [
    (64, 480, 64),   # pe block across a 64-channel boundary
    (16, 40, 32),
    (128, 96, 64),
    (3, 120, 16),
    (5, 0, 512),     # every channel rotated, 256 pairs
    (6, 60, 100),    # nope and pe/2 not multiples of 8
    (64, 384, 128),  # pe wider than 64
    (1, 6, 2),
])
def test_every_pe_placement_passes_the_shape_checks(lib, nh, nope, pe):
    """Any even pe >= 2 at any offset is a supported shape: the host checks
    pass, and without a GPU the call stops at the device check."""
    a = [k << 32 for k in range(1, 7)]  # far apart: no overlap
    for st in (lib.invrope_postmix_fwd(a[0], a[1], a[2], 8, nh, nope, pe, 0, 1e4, None),
               lib.invrope_postmix_bwd(a[0], a[1], a[2], a[3], a[4], a[5], 1 << 24,
                                       8, nh, nope, pe, 0, 1e4, None)):
        assert st not in (INVALID, UNSUPPORTED), st


def test_fwd_rejects_null_and_misaligned_pointers(lib):
    args = (8, 4, 48, 16, 0, 1e4, None)
    assert lib.invrope_postmix_fwd(None, FAKE, FAKE * 2, *args) == INVALID
    assert lib.invrope_postmix_fwd(FAKE, None, FAKE * 2, *args) == INVALID
    assert lib.invrope_postmix_fwd(FAKE, FAKE, None, *args) == INVALID
    assert lib.invrope_postmix_fwd(FAKE + 8, FAKE * 4, FAKE * 2, *args) == INVALID
    assert lib.invrope_postmix_fwd(FAKE, FAKE * 4, FAKE * 2 + 2, *args) == INVALID
    # Y overlapping O
    assert lib.invrope_postmix_fwd(FAKE, FAKE * 8, FAKE + 64, *args) == INVALID


def test_fwd_with_no_rows_is_a_no_op(lib):
    assert lib.invrope_postmix_fwd(None, None, None, 0, 4, 48, 16, 0, 1e4, None) == OK


def test_bwd_rejects_bad_arguments_on_the_host(lib):
    a = (8, 4, 48, 16, 0, 1e4, None)
    assert lib.invrope_postmix_bwd(FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6, 1 << 20,
                                   8, 4, 48, 15, 0, 1e4, None) == INVALID
    assert lib.invrope_postmix_bwd(None, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6, 1 << 20, *a) == INVALID
    assert lib.invrope_postmix_bwd(FAKE, FAKE * 2, None, FAKE * 4, FAKE * 5, FAKE * 6, 1 << 20, *a) == INVALID
    assert lib.invrope_postmix_bwd(FAKE, FAKE * 2, FAKE * 3, FAKE * 4, None, FAKE * 6, 1 << 20, *a) == INVALID
    assert lib.invrope_postmix_bwd(FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6, 1 << 20,
                                   8, 200, 448, 64, 0, 1e4, None) == UNSUPPORTED


@pytest.mark.parametrize("nh,gs,positions", [
    (4, 0, None),        # empty groups
    (4, 3, None),        # group size does not divide nh
    (4, 8, None),        # group larger than nh
    (4, 2, FAKE + 2),    # misaligned positions array
])
def test_grouped_and_positions_reject_bad_arguments(lib, nh, gs, positions):
    assert lib.invrope_postmix_fwd_ex(FAKE, FAKE * 4, FAKE * 2, 8, nh, gs, 48, 16, positions, 0, 1e4,
                                      None) == INVALID
    assert lib.invrope_postmix_bwd_ex(FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6, 1 << 20,
                                      8, nh, gs, 48, 16, positions, 0, 1e4, None) == INVALID


def test_fwd_ex_rejects_output_over_positions(lib):
    # Y = [8, 4, 64] bf16 (4 KB) starting 64 bytes before the positions array
    assert lib.invrope_postmix_fwd_ex(FAKE, FAKE * 8, FAKE * 2, 8, 4, 2, 48, 16, FAKE * 2 + 64, 0, 1e4,
                                      None) == INVALID


def test_fwd_ex_with_no_rows_is_a_no_op(lib):
    assert lib.invrope_postmix_fwd_ex(None, None, None, 0, 4, 2, 48, 16, None, 0, 1e4, None) == OK


def test_workspace_query_is_zero_for_invalid_shapes(lib):
    assert lib.invrope_postmix_bwd_workspace_bytes(8, 0, 448, 64) == 0
    assert lib.invrope_postmix_bwd_workspace_bytes(8, 4, 448, 63) == 0
    assert lib.invrope_postmix_bwd_workspace_bytes(8, 129, 448, 64) == 0


@pytest.mark.parametrize("rows,topk,sq,skv,want", [
    (10, 4, 3, 100, INVALID),          # rows not a multiple of sq
    (8, 4, 0, 100, INVALID),           # sq = 0
    (8, -1, 4, 100, INVALID),          # negative topk
    (8, 4, 4, -1, INVALID),            # negative seqlen_kv
    (8, 4, 2, 2**30, INVALID),         # 4 batches * 2^30 > 2^31
])
def test_remap_rejects_bad_arguments(lib, rows, topk, sq, skv, want):
    assert lib.kv_idx_local_to_global(FAKE, FAKE * 4, rows, topk, sq, skv, None) == want


@pytest.mark.parametrize("rows,topk,sq,skv,want", [
    (10, 4, 3, 100, INVALID),              # rows not a multiple of sq
    (8, 4, 0, 100, INVALID),               # sq = 0
    (8, 4, 4, -1, INVALID),                # negative seqlen_kv
    (8, 4, 2, 2**62, INVALID),             # 4 batches * 2^62 > 2^63
])
def test_remap_i64_rejects_bad_arguments(lib, rows, topk, sq, skv, want):
    assert lib.kv_idx_local_to_global_i64(FAKE, FAKE * 4, rows, topk, sq, skv, None) == want


def test_remap_i64_rejects_misaligned_or_overlapping_tables(lib):
    assert lib.kv_idx_local_to_global_i64(FAKE + 4, FAKE * 4, 8, 4, 4, 100, None) == INVALID
    assert lib.kv_idx_local_to_global_i64(FAKE, FAKE + 8, 8, 4, 4, 100, None) == INVALID
    assert lib.kv_idx_local_to_global_i64(None, None, 0, 16, 4, 100, None) == OK


def test_remap_empty_table_is_a_no_op(lib):
    assert lib.kv_idx_local_to_global(None, None, 0, 16, 4, 100, None) == OK
    assert lib.kv_idx_local_to_global(None, None, 8, 0, 4, 100, None) == OK


def test_remap_rejects_partial_overlap(lib):
    assert lib.kv_idx_local_to_global(FAKE, FAKE + 4, 8, 4, 4, 100, None) == INVALID


def test_binding_refuses_cpu_tensors():
    """There is no CPU fallback: host tensors are refused before any call."""
    O = torch.zeros(4, 2, 64, dtype=torch.bfloat16)
    M = torch.eye(2)
    with pytest.raises(ValueError, match="CUDA"):
        ir.invrope_postmix_fwd(O, M, 0, 48, 16)
    with pytest.raises(ValueError, match="CUDA"):
        ir.invrope_postmix_bwd(O, O, M, 0, 48, 16)
    with pytest.raises(ValueError, match="CUDA"):
        ir.kv_idx_local_to_global(torch.zeros(4, 4, dtype=torch.int32), 2, 10)


def test_binding_refuses_wrong_dtypes():
    with pytest.raises(TypeError):
        ir.invrope_postmix_fwd(torch.zeros(4, 2, 64), torch.eye(2), 0, 48, 16)
    with pytest.raises(TypeError):
        ir.kv_idx_local_to_global(torch.zeros(4, 4, dtype=torch.int64), 2, 10)


def test_watchdog_selftest_rejects_bad_limits(lib):
    v = ctypes.c_int(7)
    assert lib.invrope_watchdog_selftest(10, ctypes.byref(v)) == INVALID
    assert lib.invrope_watchdog_selftest(10**7, ctypes.byref(v)) == INVALID
    assert lib.invrope_watchdog_selftest(50000, None) == INVALID
