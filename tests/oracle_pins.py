"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each ``check_*`` takes an implementation namespace with the oracle's API and
raises ``AssertionError`` when the implementation breaks the pinned fact.
``test_oracle_pins.py`` runs them on the real oracle; ``test_oracle_mutations.py``
runs them on deliberately wrong variants to show that a plausible mistake
(a flipped sign, a wrong pairing, a transposed operand, a dropped term, a
wrong frequency or a wrong remap offset) fails at least one of them.

What pins what (the pages print no numeric example, so the pins are closed
forms, hand-derived integers, invariants and brute force):

* frequency schedule: closed forms of ``theta**(-2i/pe)`` at exact points;
* rotate-half pairing and rotation direction: the hand-derived quarter /
  half-turn example in ``golden/postmix_quarter_turns.json``;
* forward definition: pure-Python brute force on a tiny case, the position-0
  and identity / permutation special cases, commutation of the head mix with
  the per-position rotation;
* backward: pure-Python brute force of dO (both the full backward and the
  dO-only function), the adjoint identity ``<fwd(O), dY> = <O, dO(dY)>``, dM
  from unit matrices (``Y`` is linear in ``M``) and central finite differences;
* remap: the hand-derived ``golden/kv_remap_small.json`` and brute force;
  the int64 table the same, plus the 64-bit wrap;
* grouped postmix: one group equals the ungrouped postmix, several groups
  equal the ungrouped postmix with the block-diagonal matrix (and dM's
  diagonal blocks), and pure-Python brute force on a tiny case;
* folded positions: closed form, and a folded batch equals its sequences
  run one by one.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, rtol=1e-12, atol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    scale = max(1.0, float(np.max(np.abs(b)))) if b.size else 1.0
    assert err <= atol + rtol * scale, f"{what}: max|diff|={err:g}"


def _tiny_case(seed=0, sq=3, nh=3, nope=2, pe=4):
    r = _rng(seed)
    d = nope + pe
    O = r.standard_normal((sq, nh, d))
    dY = r.standard_normal((sq, nh, d))
    M = np.eye(nh) + 0.3 * r.standard_normal((nh, nh))
    pos = np.array([5, 0, 11, 2, 7, 3][:sq], dtype=np.int64)
    return O, dY, M, pos, nope, pe, 100.0


# --------------------------------------------------------------------------
# frequencies and rotation
# --------------------------------------------------------------------------

def check_inv_freq_closed_forms(impl):
    # 16 ** (-2i/8) = 2 ** (-i): exact in binary floating point
    _close(impl.inv_freq(8, 16.0), [1.0, 0.5, 0.25, 0.125], rtol=0, atol=0,
           what="inv_freq(8, 16)")
    # 10000 ** (-2/4) = 1/100
    _close(impl.inv_freq(4, 10000.0), [1.0, 0.01], rtol=1e-15, atol=0,
           what="inv_freq(4, 1e4)")
    _close(impl.inv_freq(2, 10000.0), [1.0], rtol=0, atol=0, what="inv_freq(2)")
    # the schedule is monotone decreasing and f_0 = 1 for any theta > 1
    f = impl.inv_freq(64, 10000.0)
    assert f.shape == (32,) and f[0] == 1.0 and np.all(np.diff(f) < 0)
    # last frequency of the production schedule: 10000 ** (-62/64)
    _close(f[-1], 10000.0 ** (-62.0 / 64.0), rtol=1e-15, atol=0, what="f_31")


def check_angle_is_position_at_f0(impl):
    # f_0 = 1, so the angle of pair 0 is the position in radians
    pos = np.array([0, 1, 2, 7, 32767], dtype=np.int64)
    cos, sin = impl.rope_angles(pos, 6, 500.0)
    for k, p in enumerate(pos):
        _close(cos[k, 0], math.cos(float(p)), rtol=0, atol=1e-15, what="cos p")
        _close(sin[k, 0], math.sin(float(p)), rtol=0, atol=1e-15, what="sin p")


def check_golden_quarter_turns(impl):
    g = _load("postmix_quarter_turns.json")
    O = np.array(g["O"], dtype=np.float64)
    M = np.array(g["M"], dtype=np.float64)
    dY = np.array(g["dY"], dtype=np.float64)
    pos = np.arange(g["pos0"], g["pos0"] + O.shape[0], dtype=np.int64)
    nope, pe, theta = g["nope"], g["pe"], g["theta"]
    Y = impl.postmix_fwd(O, M, pos, nope, pe, theta)
    _close(Y, g["Y"], atol=1e-12, what="golden Y")
    dO, dM = impl.postmix_bwd(dY, O, M, pos, nope, pe, theta)
    _close(dO, g["dO"], atol=1e-12, what="golden dO")
    _close(dM, g["dM"], atol=1e-12, what="golden dM")
    _close(np.sum(Y * dY), g["inner_product"], atol=1e-12, what="<Y,dY>")


def check_rope_inverts_invrope(impl):
    O, _, _, pos, nope, pe, theta = _tiny_case(1, sq=6, nh=2, nope=3, pe=8)
    X = impl.invrope(O, pos, nope, pe, theta)
    _close(impl.rope(X, pos, nope, pe, theta), O, what="rope(invrope(O))")
    _close(impl.invrope(impl.rope(O, pos, nope, pe, theta), pos, nope, pe, theta),
           O, what="invrope(rope(O))")


def check_pairs_keep_norm_and_nope_passes(impl):
    O, _, _, pos, nope, pe, theta = _tiny_case(2, sq=6, nh=3, nope=5, pe=6)
    X = impl.invrope(O, pos, nope, pe, theta)
    assert np.array_equal(X[..., :nope], O[..., :nope]), "nope channels changed"
    h = pe // 2
    n_in = O[..., nope:nope + h] ** 2 + O[..., nope + h:] ** 2
    n_out = X[..., nope:nope + h] ** 2 + X[..., nope + h:] ** 2
    _close(n_out, n_in, what="pair norms")


def check_position_zero_is_identity(impl):
    O, _, M, _, nope, pe, theta = _tiny_case(3)
    pos = np.zeros(O.shape[0], dtype=np.int64)
    assert np.array_equal(impl.invrope(O, pos, nope, pe, theta), O)
    _close(impl.postmix_fwd(O, M, pos, nope, pe, theta),
           np.einsum("gh,shc->sgc", M, O), what="pos 0")


# --------------------------------------------------------------------------
# forward
# --------------------------------------------------------------------------

def check_fwd_brute_force(impl):
    O, _, M, pos, nope, pe, theta = _tiny_case(4)
    sq, nh, d = O.shape
    h = pe // 2
    Y = np.zeros_like(O)
    for s in range(sq):
        for g in range(nh):
            for c in range(d):
                acc = 0.0
                for k in range(nh):
                    if c < nope:
                        x = O[s, k, c]
                    else:
                        i = (c - nope) % h
                        a = pos[s] * theta ** (-2.0 * i / pe)
                        x1, x2 = O[s, k, nope + i], O[s, k, nope + h + i]
                        x = (x1 * math.cos(a) + x2 * math.sin(a) if c < nope + h
                             else x2 * math.cos(a) - x1 * math.sin(a))
                    acc += M[g, k] * x
                Y[s, g, c] = acc
    _close(impl.postmix_fwd(O, M, pos, nope, pe, theta), Y, what="brute force Y")


def check_mix_commutes_with_rotation(impl):
    O, _, M, pos, nope, pe, theta = _tiny_case(5, sq=5, nh=4, nope=4, pe=8)
    Y = impl.postmix_fwd(O, M, pos, nope, pe, theta)
    # mix first (positions all 0 -> no rotation), then rotate the mixed rows
    mixed = impl.postmix_fwd(O, M, np.zeros_like(pos), nope, pe, theta)
    _close(Y, impl.invrope(mixed, pos, nope, pe, theta), what="commutation")


def check_identity_and_permutation_mix(impl):
    O, _, _, pos, nope, pe, theta = _tiny_case(6, sq=4, nh=4, nope=2, pe=4)
    X = impl.invrope(O, pos, nope, pe, theta)
    _close(impl.postmix_fwd(O, np.eye(4), pos, nope, pe, theta), X, what="M=I")
    perm = np.array([2, 0, 3, 1])
    P = np.zeros((4, 4))
    P[np.arange(4), perm] = 1.0       # Y[g] = X[perm[g]]
    _close(impl.postmix_fwd(O, P, pos, nope, pe, theta), X[:, perm, :],
           what="permutation")


# --------------------------------------------------------------------------
# backward
# --------------------------------------------------------------------------

def check_bwd_brute_force_dO(impl):
    O, dY, M, pos, nope, pe, theta = _tiny_case(7)
    sq, nh, d = O.shape
    h = pe // 2
    G = np.zeros_like(dY)
    for s in range(sq):
        for k in range(nh):
            for c in range(d):
                G[s, k, c] = sum(M[g, k] * dY[s, g, c] for g in range(nh))
    dO = G.copy()
    for s in range(sq):
        for i in range(h):
            a = pos[s] * theta ** (-2.0 * i / pe)
            g1 = G[s, :, nope + i].copy()
            g2 = G[s, :, nope + h + i].copy()
            dO[s, :, nope + i] = g1 * math.cos(a) - g2 * math.sin(a)
            dO[s, :, nope + h + i] = g2 * math.cos(a) + g1 * math.sin(a)
    got, _ = impl.postmix_bwd(dY, O, M, pos, nope, pe, theta)
    _close(got, dO, what="brute force dO")
    _close(impl.postmix_bwd_dO(dY, M, pos, nope, pe, theta), dO, what="brute force dO (dO only)")


def check_adjoint_identity(impl):
    O, dY, M, pos, nope, pe, theta = _tiny_case(8, sq=6, nh=5, nope=3, pe=6)
    Y = impl.postmix_fwd(O, M, pos, nope, pe, theta)
    dO, dM = impl.postmix_bwd(dY, O, M, pos, nope, pe, theta)
    lhs = float(np.sum(Y * dY))
    _close(float(np.sum(O * dO)), lhs, what="<fwd(O),dY> vs <O,dO>")
    _close(float(np.sum(M * dM)), lhs, what="<M,dM> (Y linear in M)")


def check_dM_from_unit_matrices(impl):
    O, dY, M, pos, nope, pe, theta = _tiny_case(9, sq=4, nh=3, nope=2, pe=4)
    nh = M.shape[0]
    _, dM = impl.postmix_bwd(dY, O, M, pos, nope, pe, theta)
    ref = np.zeros((nh, nh))
    for g in range(nh):
        for k in range(nh):
            E = np.zeros((nh, nh))
            E[g, k] = 1.0
            ref[g, k] = np.sum(impl.postmix_fwd(O, E, pos, nope, pe, theta) * dY)
    _close(dM, ref, what="dM from unit matrices")


def check_dM_finite_difference(impl):
    O, dY, M, pos, nope, pe, theta = _tiny_case(10, sq=5, nh=3, nope=3, pe=4)
    _, dM = impl.postmix_bwd(dY, O, M, pos, nope, pe, theta)
    eps = 1e-4
    for g, k in [(0, 0), (0, 2), (2, 1)]:
        Mp = M.copy()
        Mm = M.copy()
        Mp[g, k] += eps
        Mm[g, k] -= eps
        Lp = np.sum(impl.postmix_fwd(O, Mp, pos, nope, pe, theta) * dY)
        Lm = np.sum(impl.postmix_fwd(O, Mm, pos, nope, pe, theta) * dY)
        _close(dM[g, k], (Lp - Lm) / (2 * eps), rtol=1e-7, atol=1e-7,
               what=f"finite difference dM[{g},{k}]")


def check_dM_row_blocks(impl):
    O, dY, _, pos, nope, pe, theta = _tiny_case(11, sq=6, nh=2, nope=2, pe=4)
    a = impl.postmix_bwd_dM(dY, O, pos, nope, pe, theta, rows_per_chunk=1)
    b = impl.postmix_bwd_dM(dY, O, pos, nope, pe, theta, rows_per_chunk=4)
    _close(a, b, what="dM independent of row blocking")


# --------------------------------------------------------------------------
# remap
# --------------------------------------------------------------------------

def check_remap_golden(impl):
    g = _load("kv_remap_small.json")
    out = impl.kv_idx_local_to_global(np.array(g["idx"], dtype=np.int32),
                                      g["sq"], g["seqlen_kv"])
    assert out.dtype == np.int32
    assert np.array_equal(out, np.array(g["out"], dtype=np.int32)), out


def check_remap_brute_force(impl):
    r = _rng(12)
    b, sq, topk, skv = 3, 5, 7, 1000
    idx = r.integers(0, skv, size=(b * sq, topk)).astype(np.int32)
    idx[r.random(idx.shape) < 0.2] = -1
    out = impl.kv_idx_local_to_global(idx, sq, skv)
    for row in range(b * sq):
        for k in range(topk):
            v = int(idx[row, k])
            want = v if v < 0 else v + (row // sq) * skv
            assert int(out[row, k]) == want, (row, k, v, int(out[row, k]))


def check_remap_wraps_int32(impl):
    idx = np.array([[2**30], [2**30]], dtype=np.int32)
    out = impl.kv_idx_local_to_global(idx, 1, 2**30)
    # batch 1: 2^30 + 2^30 = 2^31 wraps to -2^31 in 32-bit two's complement
    assert out.tolist() == [[2**30], [-2**31]], out.tolist()


# --------------------------------------------------------------------------
# grouped postmix, arbitrary positions, int64 remap
# --------------------------------------------------------------------------

def _grouped_case(seed, sq=4, ng=2, gs=3, nope=2, pe=4):
    r = _rng(seed)
    nh = ng * gs
    O = r.standard_normal((sq, nh, nope + pe))
    dY = r.standard_normal((sq, nh, nope + pe))
    Mg = np.eye(gs)[None] + 0.3 * r.standard_normal((ng, gs, gs))
    pos = np.array([3, 0, 9, 4, 1, 6][:sq], dtype=np.int64)
    return O, dY, Mg, pos, nope, pe, 50.0


def _block_diag(Mg):
    ng, gs, _ = Mg.shape
    M = np.zeros((ng * gs, ng * gs))
    for k in range(ng):
        M[k * gs:(k + 1) * gs, k * gs:(k + 1) * gs] = Mg[k]
    return M


def check_grouped_one_group_is_ungrouped(impl):
    O, dY, M, pos, nope, pe, theta = _tiny_case(13)
    _close(impl.postmix_fwd_grouped(O, M[None], pos, nope, pe, theta),
           impl.postmix_fwd(O, M, pos, nope, pe, theta), what="one group: Y")
    dO_g, dM_g = impl.postmix_bwd_grouped(dY, O, M[None], pos, nope, pe, theta)
    dO, dM = impl.postmix_bwd(dY, O, M, pos, nope, pe, theta)
    _close(dO_g, dO, what="one group: dO")
    _close(dM_g[0], dM, what="one group: dM")


def check_grouped_is_block_diagonal_mix(impl):
    O, dY, Mg, pos, nope, pe, theta = _grouped_case(14)
    M = _block_diag(Mg)
    _close(impl.postmix_fwd_grouped(O, Mg, pos, nope, pe, theta),
           impl.postmix_fwd(O, M, pos, nope, pe, theta), what="grouped Y")
    dO_g, dM_g = impl.postmix_bwd_grouped(dY, O, Mg, pos, nope, pe, theta)
    dO, dM = impl.postmix_bwd(dY, O, M, pos, nope, pe, theta)
    _close(dO_g, dO, what="grouped dO")
    gs = Mg.shape[1]
    for k in range(Mg.shape[0]):
        sl = slice(k * gs, (k + 1) * gs)
        _close(dM_g[k], dM[sl, sl], what=f"grouped dM block {k}")


def check_grouped_brute_force(impl):
    O, dY, Mg, pos, nope, pe, theta = _grouped_case(15, sq=2, ng=2, gs=2, nope=1, pe=2)
    sq, nh, d = O.shape
    gs = Mg.shape[1]
    X = np.zeros_like(O)
    for s in range(sq):
        a = pos[s] * 1.0          # pe = 2: one pair, f_0 = 1, angle = position
        for h in range(nh):
            X[s, h, 0] = O[s, h, 0]
            X[s, h, 1] = O[s, h, 1] * math.cos(a) + O[s, h, 2] * math.sin(a)
            X[s, h, 2] = O[s, h, 2] * math.cos(a) - O[s, h, 1] * math.sin(a)
    Y = np.zeros_like(O)
    dM = np.zeros_like(Mg)
    for s in range(sq):
        for g in range(nh):
            k, i = divmod(g, gs)
            for c in range(d):
                Y[s, g, c] = sum(Mg[k, i, j] * X[s, k * gs + j, c] for j in range(gs))
                for j in range(gs):
                    dM[k, i, j] += dY[s, g, c] * X[s, k * gs + j, c]
    # dO: the group's transposed mix of dY, rotated back by +a (pe = 2: one pair)
    dO = np.zeros_like(O)
    for s in range(sq):
        a = pos[s] * 1.0
        for h in range(nh):
            k, j = divmod(h, gs)
            G = [sum(Mg[k, i, j] * dY[s, k * gs + i, c] for i in range(gs)) for c in range(d)]
            dO[s, h, 0] = G[0]
            dO[s, h, 1] = G[1] * math.cos(a) - G[2] * math.sin(a)
            dO[s, h, 2] = G[2] * math.cos(a) + G[1] * math.sin(a)
    _close(impl.postmix_fwd_grouped(O, Mg, pos, nope, pe, theta), Y, what="brute force grouped Y")
    got_dO, got_dM = impl.postmix_bwd_grouped(dY, O, Mg, pos, nope, pe, theta)
    _close(got_dM, dM, what="brute force grouped dM")
    _close(got_dO, dO, what="brute force grouped dO")
    _close(impl.postmix_bwd_grouped_dO(dY, Mg, pos, nope, pe, theta), dO,
           what="brute force grouped dO (dO only)")


def check_positions_batched(impl):
    assert impl.positions_batched(3, 4, 10).tolist() == [10, 11, 12, 13] * 3
    assert impl.positions_batched(1, 5).tolist() == [0, 1, 2, 3, 4]
    # folded sequences rotate like the same rows run one sequence at a time
    O, _, M, _, nope, pe, theta = _tiny_case(16, sq=6, nh=2, nope=2, pe=4)
    pos = impl.positions_batched(2, 3, 7)
    Y = impl.postmix_fwd(O, M, pos, nope, pe, theta)
    for b in range(2):
        rows = slice(3 * b, 3 * b + 3)
        _close(Y[rows], impl.postmix_fwd(O[rows], M, impl.positions_contiguous(3, 7), nope, pe, theta),
               what=f"batch {b}")


def check_remap_i64_brute_force(impl):
    r = _rng(17)
    b, sq, topk, skv = 3, 4, 5, 3 * 2**40
    idx = r.integers(0, skv, size=(b * sq, topk)).astype(np.int64)
    idx[r.random(idx.shape) < 0.2] = -7
    out = impl.kv_idx_local_to_global_i64(idx, sq, skv)
    assert out.dtype == np.int64
    for row in range(b * sq):
        for k in range(topk):
            v = int(idx[row, k])
            want = v if v < 0 else v + (row // sq) * skv
            assert int(out[row, k]) == want, (row, k, v, int(out[row, k]))


def check_remap_i64_wraps_and_matches_i32(impl):
    out = impl.kv_idx_local_to_global_i64(np.array([[2**62], [2**62]], dtype=np.int64), 1, 2**62)
    # batch 1: 2^62 + 2^62 = 2^63 wraps to -2^63 in 64-bit two's complement
    assert out.tolist() == [[2**62], [-2**63]], out.tolist()
    g = _load("kv_remap_small.json")
    idx = np.array(g["idx"], dtype=np.int64)
    assert impl.kv_idx_local_to_global_i64(idx, g["sq"], g["seqlen_kv"]).tolist() == g["out"]


ALL_CHECKS = [
    check_inv_freq_closed_forms,
    check_angle_is_position_at_f0,
    check_golden_quarter_turns,
    check_rope_inverts_invrope,
    check_pairs_keep_norm_and_nope_passes,
    check_position_zero_is_identity,
    check_fwd_brute_force,
    check_mix_commutes_with_rotation,
    check_identity_and_permutation_mix,
    check_bwd_brute_force_dO,
    check_adjoint_identity,
    check_dM_from_unit_matrices,
    check_dM_finite_difference,
    check_dM_row_blocks,
    check_remap_golden,
    check_remap_brute_force,
    check_remap_wraps_int32,
    check_grouped_one_group_is_ungrouped,
    check_grouped_is_block_diagonal_mix,
    check_grouped_brute_force,
    check_positions_batched,
    check_remap_i64_brute_force,
    check_remap_i64_wraps_and_matches_i32,
]
