"""The debug-bounds build (device-side index checks, ``build.py --debug-bounds``)
runs the forward, the backward (block-diagonal, stacked and 128-channel
kernels), the grouped mix, per-row positions and the remap in a fresh process
and records no fault code. Needs a GB300 (sm_103a)."""

import os
import subprocess
import sys
import textwrap

import pytest

from partial_inverse_rope_gb300.build import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import torch
    import partial_inverse_rope_gb300 as ir
    from partial_inverse_rope_gb300 import inputs as W

    shapes = [(128, 4, 48, 16), (37, 3, 56, 8), (257, 64, 448, 64), (301, 64, 480, 32),
              (70, 100, 448, 64), (33, 128, 448, 64), (65, 1, 448, 64), (40, 128, 64, 64),
              (300, 64, 480, 64), (77, 128, 96, 64), (33, 6, 60, 100), (45, 5, 0, 512), (70, 12, 62, 10)]
    for sq, nh, nope, pe in shapes:
        O = W.normal_bf16((sq, nh, nope + pe), 1, "cuda")
        dY = W.normal_bf16((sq, nh, nope + pe), 2, "cuda")
        M = W.postmix_M(nh, 3, "cuda")
        ir.invrope_postmix_fwd(O, M, 5, nope, pe)
        ir.invrope_postmix_bwd(dY, O, M, 5, nope, pe)
    O = W.normal_bf16((130, 64, 512), 4, "cuda")
    dY = W.normal_bf16((130, 64, 512), 5, "cuda")
    Mg = W.postmix_Mg(8, 8, 6, "cuda")
    pos = W.random_positions(130, 7, 0, 1 << 20, "cuda")
    ir.invrope_postmix_fwd_ex(O, Mg, 448, 64, positions=pos, group_size=8)
    ir.invrope_postmix_bwd_ex(dY, O, Mg, 448, 64, positions=pos, group_size=8)
    idx = torch.randint(-1, 1000, (4 * 64, 40), dtype=torch.int32, device="cuda")
    ir.kv_idx_local_to_global(idx, 64, 1000)
    ir.kv_idx_local_to_global_i64(idx.to(torch.int64), 64, 1000)
    code = ir.invrope_take_device_fault()
    print("debug-bounds fault code", hex(code))
    assert code == 0, hex(code)
""")


def test_debug_bounds_build_records_no_fault():
    lib = build(debug_bounds=True)
    env = dict(os.environ, INVROPE_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-c", SCRIPT], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "fault code 0x0" in r.stdout
