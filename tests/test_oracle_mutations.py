"""Plant plausible mistakes in copies of the oracle and show the pins catch them.

Every mutant below is the oracle with exactly one deliberate error. The test
passes only if at least one pin in ``oracle_pins.ALL_CHECKS`` fails on it, so a
pin set that would let such a mistake through is itself a test failure.
"""

import types

import numpy as np
import pytest

import oracle
from oracle import invrope_oracle as base
from oracle_pins import ALL_CHECKS


def _namespace(**overrides):
    ns = {name: getattr(base, name) for name in base.__all__}
    ns.update(overrides)
    return types.SimpleNamespace(**ns)


def _rotate_with(sign_inv, pairing="half", freq=None):
    """Build (invrope, rope) with a chosen inverse sign, pairing and schedule."""
    def angles(positions, pe, theta):
        f = base.inv_freq(pe, theta) if freq is None else freq(pe, theta)
        a = np.asarray(positions, dtype=np.float64)[:, None] * f[None, :]
        return np.cos(a), np.sin(a)

    def rot(x, positions, nope, pe, theta, sign):
        x = np.asarray(x, dtype=np.float64)
        cos, sin = angles(positions, pe, theta)
        out = x.copy()
        h = pe // 2
        if pairing == "half":
            i1 = nope + np.arange(h)
            i2 = i1 + h
        else:  # interleaved pairs (nope+2i, nope+2i+1)
            i1 = nope + 2 * np.arange(h)
            i2 = i1 + 1
        c = cos[:, None, :]
        s = sign * sin[:, None, :]
        x1, x2 = x[:, :, i1], x[:, :, i2]
        out[:, :, i1] = x1 * c - x2 * s
        out[:, :, i2] = x2 * c + x1 * s
        return out

    def inv(x, positions, nope, pe, theta):
        return rot(x, positions, nope, pe, theta, sign_inv)

    def fwd_rope(x, positions, nope, pe, theta):
        return rot(x, positions, nope, pe, theta, -sign_inv)

    return inv, fwd_rope, angles


def _postmix_ns(inv, fwd_rope, angles, mix_t=False, bwd_M=False, drop_nope=False,
                dM_t=False, bwd_rot=None):
    def postmix_fwd(O, M, positions, nope, pe, theta):
        X = inv(O, positions, nope, pe, theta)
        if drop_nope:
            X[..., :nope] = 0.0
        M = np.asarray(M, dtype=np.float64)
        return np.matmul((M.T if mix_t else M)[None], X)

    def postmix_bwd_dM(dY, O, positions, nope, pe, theta, rows_per_chunk=512):
        X = inv(O, positions, nope, pe, theta)
        if drop_nope:
            X[..., :nope] = 0.0
        dM = np.einsum("sgc,shc->gh", np.asarray(dY, dtype=np.float64), X)
        return dM.T if dM_t else dM

    def postmix_bwd_dO(dY, M, positions, nope, pe, theta):
        M = np.asarray(M, dtype=np.float64)
        G = np.matmul((M if bwd_M else M.T)[None], np.asarray(dY, dtype=np.float64))
        rot = fwd_rope if bwd_rot is None else bwd_rot
        return rot(G, positions, nope, pe, theta)

    def postmix_bwd(dY, O, M, positions, nope, pe, theta):
        dO = postmix_bwd_dO(dY, M, positions, nope, pe, theta)
        return dO, postmix_bwd_dM(dY, O, positions, nope, pe, theta)

    return _namespace(invrope=inv, rope=fwd_rope, rope_angles=angles,
                      postmix_fwd=postmix_fwd, postmix_bwd=postmix_bwd,
                      postmix_bwd_dO=postmix_bwd_dO, postmix_bwd_dM=postmix_bwd_dM)


def _mutants():
    ok_inv, ok_rope, ok_angles = _rotate_with(-1.0)
    bad_inv, bad_rope, _ = _rotate_with(+1.0)
    il_inv, il_rope, il_angles = _rotate_with(-1.0, pairing="interleaved")

    def freq_shift(pe, theta):
        i = np.arange(pe // 2, dtype=np.float64)
        return np.power(float(theta), -2.0 * (i + 1) / pe)

    def freq_half(pe, theta):
        i = np.arange(pe // 2, dtype=np.float64)
        return np.power(float(theta), -1.0 * i / pe)

    fs_inv, fs_rope, fs_angles = _rotate_with(-1.0, freq=freq_shift)
    fh_inv, fh_rope, fh_angles = _rotate_with(-1.0, freq=freq_half)

    def remap_by_row(idx, sq, seqlen_kv):
        idx = np.asarray(idx).astype(np.int64)
        r = np.arange(idx.shape[0])[:, None]
        return np.where(idx >= 0, idx + r * seqlen_kv, idx).astype(np.int32)

    def remap_shifts_padding(idx, sq, seqlen_kv):
        idx = np.asarray(idx).astype(np.int64)
        b = (np.arange(idx.shape[0]) // sq)[:, None]
        return (idx + b * seqlen_kv).astype(np.int32)

    def remap_no_wrap(idx, sq, seqlen_kv):
        idx = np.asarray(idx).astype(np.int64)
        b = (np.arange(idx.shape[0]) // sq)[:, None]
        out = np.where(idx >= 0, idx + b * seqlen_kv, idx)
        return np.clip(out, -2**31, 2**31 - 1).astype(np.int32)

    def grouped_ns(transpose_fwd=False, strided=False, dM_t=False, dO_mix_untransposed=False):
        def groups(nh, gs):
            ng = nh // gs
            if strided:  # heads k, k+ng, k+2ng, ... instead of consecutive heads
                return [np.arange(k, nh, ng) for k in range(ng)]
            return [np.arange(k * gs, (k + 1) * gs) for k in range(ng)]

        def fwd(O, Mg, positions, nope, pe, theta):
            X = base.invrope(O, positions, nope, pe, theta)
            Mg = np.asarray(Mg, dtype=np.float64)
            Y = np.empty_like(X)
            for k, hs in enumerate(groups(X.shape[1], Mg.shape[1])):
                m = Mg[k].T if transpose_fwd else Mg[k]
                Y[:, hs, :] = np.matmul(m[None], X[:, hs, :])
            return Y

        def bwd_dO(dY, Mg, positions, nope, pe, theta):
            Mg = np.asarray(Mg, dtype=np.float64)
            dY = np.asarray(dY, dtype=np.float64)
            G = np.empty_like(dY)
            for k, hs in enumerate(groups(dY.shape[1], Mg.shape[1])):
                m = Mg[k] if dO_mix_untransposed else Mg[k].T
                G[:, hs, :] = np.matmul(m[None], dY[:, hs, :])
            return base.rope(G, positions, nope, pe, theta)

        def bwd(dY, O, Mg, positions, nope, pe, theta):
            Mg = np.asarray(Mg, dtype=np.float64)
            dY = np.asarray(dY, dtype=np.float64)
            X = base.invrope(O, positions, nope, pe, theta)
            dM = np.empty_like(Mg)
            for k, hs in enumerate(groups(dY.shape[1], Mg.shape[1])):
                blk = np.einsum("sgc,shc->gh", dY[:, hs, :], X[:, hs, :])
                dM[k] = blk.T if dM_t else blk
            return bwd_dO(dY, Mg, positions, nope, pe, theta), dM

        return _namespace(postmix_fwd_grouped=fwd, postmix_bwd_grouped=bwd, postmix_bwd_grouped_dO=bwd_dO)

    def remap64_by_row(idx, sq, seqlen_kv):
        idx = np.asarray(idx).astype(np.int64)
        r = np.arange(idx.shape[0])[:, None]
        return np.where(idx >= 0, idx + r * seqlen_kv, idx)

    def remap64_saturates(idx, sq, seqlen_kv):
        idx = np.asarray(idx).astype(object)
        b = (np.arange(idx.shape[0]) // sq)[:, None]
        out = np.where(idx >= 0, idx + b * int(seqlen_kv), idx)
        return np.clip(out, -2**63, 2**63 - 1).astype(np.int64)

    def remap64_via_int32(idx, sq, seqlen_kv):
        return base.kv_idx_local_to_global(np.asarray(idx).astype(np.int32), sq, seqlen_kv).astype(np.int64)

    return {
        "grouped_blocks_transposed": grouped_ns(transpose_fwd=True),
        "grouped_heads_strided": grouped_ns(strided=True),
        "grouped_dM_transposed": grouped_ns(dM_t=True),
        "grouped_dO_mix_untransposed": grouped_ns(dO_mix_untransposed=True),
        "remap64_offset_by_row": _namespace(kv_idx_local_to_global_i64=remap64_by_row),
        "remap64_saturates": _namespace(kv_idx_local_to_global_i64=remap64_saturates),
        "remap64_truncates_to_int32": _namespace(kv_idx_local_to_global_i64=remap64_via_int32),
        "inverse_rotates_forward": _postmix_ns(bad_inv, bad_rope, ok_angles),
        "interleaved_pairs": _postmix_ns(il_inv, il_rope, il_angles),
        "frequency_index_shift": _postmix_ns(fs_inv, fs_rope, fs_angles),
        "frequency_exponent_halved": _postmix_ns(fh_inv, fh_rope, fh_angles),
        "mix_transposed": _postmix_ns(ok_inv, ok_rope, ok_angles, mix_t=True),
        "bwd_uses_M_not_MT": _postmix_ns(ok_inv, ok_rope, ok_angles, bwd_M=True),
        "nope_dropped": _postmix_ns(ok_inv, ok_rope, ok_angles, drop_nope=True),
        "dM_transposed": _postmix_ns(ok_inv, ok_rope, ok_angles, dM_t=True),
        "dO_rotates_backwards": _postmix_ns(ok_inv, ok_rope, ok_angles,
                                            bwd_rot=ok_inv),
        "remap_offset_by_row": _namespace(kv_idx_local_to_global=remap_by_row),
        "remap_shifts_padding": _namespace(kv_idx_local_to_global=remap_shifts_padding),
        "remap_saturates": _namespace(kv_idx_local_to_global=remap_no_wrap),
    }


MUTANTS = _mutants()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    impl = MUTANTS[name]
    failed = []
    for check in ALL_CHECKS:
        try:
            check(impl)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, f"no pin caught the planted mistake '{name}'"


def test_unmutated_namespace_passes_everything():
    inv, rot, ang = _rotate_with(-1.0)
    impl = _postmix_ns(inv, rot, ang)
    for check in ALL_CHECKS:
        check(impl)
    for check in ALL_CHECKS:
        check(oracle)
