"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
binding and the fp64 oracle on the same seeded inputs, and compare."""

from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from partial_inverse_rope_gb300 import binding
from partial_inverse_rope_gb300.build import build
from partial_inverse_rope_gb300.inputs import normal_bf16, postmix_M

# Tolerances (written here, applied element by element):
#   bf16 outputs Y / dO:  max |gpu - oracle| <= 8e-3 * max |oracle|
#   fp32 dM:              ||gpu - oracle||_F / ||oracle||_F <= 1e-4
BF16_TOL = 8e-3
DM_TOL = 1e-4


def ensure_built():
    if not os.path.exists(binding.lib_path()):
        build()
    binding.lib()


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a bf16 / fp32 tensor to a float64 numpy array."""
    return t.detach().cpu().to(torch.float64).numpy()


def make_inputs(sq, nh, nope, pe, seed=0, device="cuda"):
    d = nope + pe
    O = normal_bf16((sq, nh, d), seed, device)
    dY = normal_bf16((sq, nh, d), seed + 1, device)
    M = postmix_M(nh, seed + 2, device)
    return O, dY, M


def bf16_err(gpu: np.ndarray, ref: np.ndarray):
    """(max |diff|, allowed) for the bf16 gate."""
    err = float(np.max(np.abs(gpu - ref))) if ref.size else 0.0
    return err, BF16_TOL * float(np.max(np.abs(ref))) if ref.size else 0.0


def assert_bf16_close(gpu: np.ndarray, ref: np.ndarray, what: str):
    err, allowed = bf16_err(gpu, ref)
    assert err <= allowed, f"{what}: max|diff| {err:.4g} > {allowed:.4g}"


def assert_dm_close(gpu: np.ndarray, ref: np.ndarray, what="dM"):
    rel = float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-300))
    assert rel <= DM_TOL, f"{what}: relative Frobenius error {rel:.3g} > {DM_TOL}"
    return rel


def compare_all_rows(O, dY, M, Y, dO, positions, nope, pe, theta, block=512, group_size=None):
    """Y and dO of the CUDA path against the oracle on every row, ``block``
    rows at a time (host memory stays bounded); ``positions`` holds the
    absolute position of every row. With ``group_size`` the mix is grouped."""
    sq = O.shape[0]
    Oc, dYc, Yc, dOc = (t.detach().cpu() for t in (O, dY, Y, dO))
    M64 = f64(M)
    for s0 in range(0, sq, block):
        s1 = min(sq, s0 + block)
        O_b, dY_b = f64(Oc[s0:s1]), f64(dYc[s0:s1])
        pos = positions[s0:s1]
        if group_size is None:
            Y_ref = oracle.postmix_fwd(O_b, M64, pos, nope, pe, theta)
            dO_ref = oracle.postmix_bwd_dO(dY_b, M64, pos, nope, pe, theta)
        else:
            Y_ref = oracle.postmix_fwd_grouped(O_b, M64, pos, nope, pe, theta)
            dO_ref = oracle.postmix_bwd_grouped_dO(dY_b, M64, pos, nope, pe, theta)
        assert_bf16_close(f64(Yc[s0:s1]), Y_ref, f"Y rows {s0}..{s1 - 1}")
        assert_bf16_close(f64(dOc[s0:s1]), dO_ref, f"dO rows {s0}..{s1 - 1}")


def oracle_fwd_rows(O_cpu64, M64, rows, pos0, nope, pe, theta):
    """Oracle Y for the given rows (positions pos0 + rows)."""
    pos = pos0 + np.asarray(rows, dtype=np.int64)
    return oracle.postmix_fwd(O_cpu64, M64, pos, nope, pe, theta)


def sample_rows(sq, P, n_random=48, seed=0):
    """First/last rows, rows around tile boundaries (P positions per tile) and random rows."""
    r = np.random.default_rng(seed)
    picks = {0, 1, sq - 1, sq - 2}
    for t in (1, 2, 3, (sq // P) // 2, sq // P - 1, sq // P):
        for dlt in (-1, 0, 1):
            s = t * P + dlt
            if 0 <= s < sq:
                picks.add(s)
    picks.update(int(x) for x in r.integers(0, sq, size=n_random))
    return np.array(sorted(picks), dtype=np.int64)
