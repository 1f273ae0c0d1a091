"""Plain fp64 reference (the oracle) for the fused HCA inverse RoPE + VHA postmix
and for the per-batch-local -> flat-global sparse-attention KV index remap.

TEST INFRASTRUCTURE: this module is the parity oracle. It is slow on purpose
and follows the definitions literally; only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline / reference
legs) may call it. The CUDA library never imports it, and it imports nothing
from the CUDA library.

Sources (web pages; cited by title and section):

* [PR1772] PaddleFleet pull request #1772, "Fuse HCA inverse RoPE into the VHA
  postmix, and the sparse-attention KV index remap".
  - English description, item 1 ``fuse_inv_rope_into_vha_postmix``: RoPE only
    touches the trailing ``qk_pos_emb_head_dim`` (= pe) channels of each head,
    the ungrouped VHA postmix is an [nh, nh] GEMM that contracts the head
    axis, so the channel axis is a pure N dimension of that GEMM.
  - Chinese description, section 1: the same statement, plus the weight
    gradient ``dM[h,h'] = sum_{t,c} dOut[t,h,c] * O_roped[t,h',c]`` that
    contracts over all tokens and the full channel axis.
  - Revision note: the backward rebuilds the full-width rotated tensor and
    hands both gradients to the matmul backward, i.e. the activation
    gradient is the GEMM's input gradient pushed back through the rotation.
  - English description item 2 / Chinese description section 2
    ``sparse_attn_global_kv_idx_remap_fusion``: the local -> global KV column
    remap ``idx + b * seqlen_kv`` over a ``[b*sq, topk]`` table, defined by the
    eager chain full + greater_equal + arange + expand + scale + add + where.

Readings where the pages are silent (each pinned by a closed-form test in
``tests/test_oracle_pins.py``, not by the pages, which print no numbers):

* rotate-half RoPE layout: pe channels ``[nope, nope+pe)``, pair ``i`` is
  ``(nope+i, nope+i+pe/2)`` for ``i < pe/2``;
* frequencies ``f_i = theta ** (-2 i / pe)``; the angle at position p is
  ``a = p * f_i``;
* RoPE rotates a pair by ``+a``: ``(x1, x2) -> (x1 cos a - x2 sin a,
  x2 cos a + x1 sin a)``; the inverse RoPE rotates by ``-a``;
* ``X = invrope(O)`` is NOT rounded to bf16 (exact real-valued operand);
* the remap keeps every negative entry (padding) unchanged and adds the batch
  offset to every non-negative entry, wrapping in 32-bit two's complement.

Array conventions: ``O, dY, Y, dO`` are ``[sq, nh, d]`` with ``d = nope+pe``
(channel fastest); ``M, dM`` are ``[nh, nh]`` with ``Y[s, g] = sum_h M[g, h]
X[s, h]``; ``positions`` is an integer array of length ``sq`` holding the
absolute position of each row (contiguous ``pos0 + s`` for the configs, or
any integers: several folded sequences, a context-parallel rebalance). The
grouped postmix takes ``Mg`` as ``[nh/gs, gs, gs]``.
"""

from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def inv_freq(pe: int, theta: float) -> np.ndarray:
    """Rotary frequencies ``f_i = theta**(-2i/pe)`` for ``i < pe/2`` (fp64).

    The pages name the rotated width ``qk_pos_emb_head_dim`` ([PR1772] item 1)
    but not the frequency schedule; this is the standard rotary schedule.
    """
    if pe < 2 or pe % 2:
        raise ValueError("pe must be a positive even number")
    i = np.arange(pe // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * i / pe)


def rope_angles(positions, pe: int, theta: float):
    """``(cos a, sin a)`` with ``a[s, i] = positions[s] * f_i``, shapes ``[sq, pe/2]``."""
    p = np.asarray(positions, dtype=np.int64).astype(np.float64)
    a = p[:, None] * inv_freq(pe, theta)[None, :]
    return np.cos(a), np.sin(a)


def _rotate(x, cos, sin, nope: int, pe: int, sign: float) -> np.ndarray:
    """Rotate every rotate-half pair of the pe channels by ``sign * a``.

    ``x`` is ``[sq, nh, d]``; ``cos``/``sin`` are ``[sq, pe/2]`` and apply to
    every head of a row (the rotation depends on the position only).
    """
    x = _f64(x)
    half = pe // 2
    out = x.copy()
    c = cos[:, None, :]
    s = sign * sin[:, None, :]
    x1 = x[:, :, nope:nope + half]
    x2 = x[:, :, nope + half:nope + pe]
    out[:, :, nope:nope + half] = x1 * c - x2 * s
    out[:, :, nope + half:nope + pe] = x2 * c + x1 * s
    return out


def invrope(x, positions, nope: int, pe: int, theta: float) -> np.ndarray:
    """Inverse RoPE on the trailing pe channels: rotate each pair by ``-a``.

    [PR1772] item 1: only the trailing ``qk_pos_emb_head_dim`` channels are
    touched; the ``nope`` leading channels pass through unchanged.
    """
    cos, sin = rope_angles(positions, pe, theta)
    return _rotate(x, cos, sin, nope, pe, -1.0)


def rope(x, positions, nope: int, pe: int, theta: float) -> np.ndarray:
    """RoPE on the trailing pe channels: rotate each pair by ``+a``.

    The rotation is orthogonal, so this is both the inverse and the adjoint
    of :func:`invrope`; the backward uses it to push the GEMM's input
    gradient back through the inverse rotation ([PR1772] revision note).
    """
    cos, sin = rope_angles(positions, pe, theta)
    return _rotate(x, cos, sin, nope, pe, +1.0)


def postmix_fwd(O, M, positions, nope: int, pe: int, theta: float) -> np.ndarray:
    """``Y[s, g, :] = sum_h M[g, h] * invrope_s(O[s, h, :])`` in fp64.

    [PR1772] item 1 / Chinese section 1: the inverse RoPE output feeds the
    ungrouped [nh, nh] postmix GEMM that contracts the head axis. The oracle
    materialises the rotated tensor on purpose (it is the unfused definition).
    """
    X = invrope(O, positions, nope, pe, theta)
    M = _f64(M)
    # contract the head axis: Y[s] = M @ X[s]   (X[s] is [nh, d])
    return np.matmul(M[None, :, :], X)


def postmix_bwd_dM(dY, O, positions, nope: int, pe: int, theta: float,
                   rows_per_chunk: int = 512) -> np.ndarray:
    """``dM[g, h] = sum_{s, c} dY[s, g, c] * X[s, h, c]`` with ``X = invrope(O)``.

    [PR1772] Chinese section 1 prints this weight gradient (with ``t`` for the
    token and ``h, h'`` for the output / input head). The sum over ``s`` is
    taken row block by row block (a block of consecutive positions per
    matmul) so that the fp64 copy of a 1 GiB bf16 tensor never exists whole.
    """
    dY = np.asarray(dY)
    O = np.asarray(O)
    sq, nh, d = dY.shape
    positions = np.asarray(positions, dtype=np.int64)
    dM = np.zeros((nh, nh), dtype=np.float64)
    for s0 in range(0, sq, rows_per_chunk):
        s1 = min(sq, s0 + rows_per_chunk)
        X = invrope(O[s0:s1], positions[s0:s1], nope, pe, theta)
        G = _f64(dY[s0:s1])
        # sum over (s, c) of G[s, g, c] * X[s, h, c]
        Gm = G.transpose(1, 0, 2).reshape(nh, -1)
        Xm = X.transpose(1, 0, 2).reshape(nh, -1)
        dM += Gm @ Xm.T
    return dM


def postmix_bwd_dO(dY, M, positions, nope: int, pe: int, theta: float) -> np.ndarray:
    """Input gradient of :func:`postmix_fwd` in fp64.

    ``dX[s, h, :] = sum_g M[g, h] dY[s, g, :]`` is the GEMM's input gradient
    and ``dO = rope(dX)`` on the pe channels (``dX`` on the nope channels)
    because the inverse rotation is orthogonal ([PR1772] revision note: the
    input gradient is the matmul backward of the unfused postmix, pushed
    through the rotation).
    """
    M = _f64(M)
    G = np.matmul(M.T[None, :, :], _f64(dY))
    return rope(G, positions, nope, pe, theta)


def postmix_bwd(dY, O, M, positions, nope: int, pe: int, theta: float):
    """Backward of :func:`postmix_fwd`: returns ``(dO, dM)`` in fp64, ``dO``
    from :func:`postmix_bwd_dO` and ``dM`` from :func:`postmix_bwd_dM`."""
    dO = postmix_bwd_dO(dY, M, positions, nope, pe, theta)
    dM = postmix_bwd_dM(dY, O, positions, nope, pe, theta)
    return dO, dM


def _group_slices(nh: int, gs: int):
    """Head slices of the groups: group ``k`` holds heads ``k*gs .. k*gs+gs-1``."""
    if gs < 1 or nh % gs:
        raise ValueError("the group size must divide nh")
    return [slice(k * gs, (k + 1) * gs) for k in range(nh // gs)]


def postmix_fwd_grouped(O, Mg, positions, nope: int, pe: int, theta: float) -> np.ndarray:
    """Grouped VHA postmix after the inverse RoPE, in fp64.

    [PR1772] Chinese description section 1 and [PR1843] list
    ``vha_postmix_grouped=True`` among the configurations the fused path
    leaves to the unfused code; the pages do not spell the grouped mix out.
    Reading: the heads form ``ng = nh / gs`` groups of ``gs`` consecutive
    heads, and each group is mixed by its own ``[gs, gs]`` matrix:
    ``Y[s, k*gs + i, :] = sum_j Mg[k, i, j] * X[s, k*gs + j, :]``, i.e. the
    ungrouped postmix with a block-diagonal head mix. ``Mg`` is
    ``[ng, gs, gs]``.
    """
    X = invrope(O, positions, nope, pe, theta)
    Mg = _f64(Mg)
    ng, gs, gs2 = Mg.shape
    if gs != gs2 or X.shape[1] != ng * gs:
        raise ValueError("Mg must be [nh/gs, gs, gs]")
    Y = np.empty_like(X)
    for k, sl in enumerate(_group_slices(X.shape[1], gs)):
        Y[:, sl, :] = np.matmul(Mg[k][None, :, :], X[:, sl, :])
    return Y


def postmix_bwd_grouped(dY, O, Mg, positions, nope: int, pe: int, theta: float):
    """Backward of :func:`postmix_fwd_grouped`: returns ``(dO, dMg)`` in fp64.

    Per group ``k``: the input gradient ``dX = Mg[k]^T dY`` on the group's
    heads, rotated back by ``+a`` on the pe channels (as in
    :func:`postmix_bwd`), and ``dMg[k, i, j] = sum_{s, c} dY[s, k*gs+i, c] *
    X[s, k*gs+j, c]`` (the weight gradient of [PR1772] Chinese section 1
    restricted to the pairs of heads that the group's matrix mixes).
    """
    Mg = _f64(Mg)
    ng, gs, _ = Mg.shape
    dY = np.asarray(dY)
    O = np.asarray(O)
    dMg = np.empty((ng, gs, gs), dtype=np.float64)
    for k, sl in enumerate(_group_slices(dY.shape[1], gs)):
        dMg[k] = postmix_bwd_dM(dY[:, sl, :], O[:, sl, :], positions, nope, pe, theta)
    dO = postmix_bwd_grouped_dO(dY, Mg, positions, nope, pe, theta)
    return dO, dMg


def postmix_bwd_grouped_dO(dY, Mg, positions, nope: int, pe: int, theta: float) -> np.ndarray:
    """Input gradient of :func:`postmix_fwd_grouped` in fp64: per group ``k``,
    ``dX = Mg[k]^T dY`` on the group's heads, rotated back by ``+a`` on the
    pe channels (as in :func:`postmix_bwd_dO`)."""
    Mg = _f64(Mg)
    dY = np.asarray(dY)
    G = np.empty(dY.shape, dtype=np.float64)
    for k, sl in enumerate(_group_slices(dY.shape[1], Mg.shape[1])):
        G[:, sl, :] = np.matmul(Mg[k].T[None, :, :], _f64(dY[:, sl, :]))
    return rope(G, positions, nope, pe, theta)


def kv_idx_local_to_global(idx, sq: int, seqlen_kv: int) -> np.ndarray:
    """Per-batch-local -> flat-global KV column indices, int32 ``[rows, topk]``.

    [PR1772] item 2 / Chinese section 2: ``out = idx + b * seqlen_kv`` where
    ``b = r // sq`` is the batch of table row ``r``; entries ``< 0`` are
    padding and pass through (the eager chain's ``greater_equal`` + ``where``).
    The addition is done in int64 and wrapped to int32 two's complement,
    which is what an int32 elementwise add produces.
    """
    idx = np.asarray(idx)
    if idx.ndim != 2:
        raise ValueError("idx must be [rows, topk]")
    rows = idx.shape[0]
    if sq <= 0 or rows % sq:
        raise ValueError("rows must be a multiple of sq")
    b = np.arange(rows, dtype=np.int64) // sq
    wide = idx.astype(np.int64)
    shifted = wide + (b * int(seqlen_kv))[:, None]
    out = np.where(wide >= 0, shifted, wide)
    return ((out + 2**31) % 2**32 - 2**31).astype(np.int32)


def kv_idx_local_to_global_i64(idx, sq: int, seqlen_kv: int) -> np.ndarray:
    """The remap of :func:`kv_idx_local_to_global` on an int64 table.

    [PR1772] (the note on the remap tests' host memory) builds the remap
    tables once per index dtype, with topk widths 640 and 2176. Same rule:
    ``out = idx + (r // sq) * seqlen_kv`` where ``idx >= 0``, padding
    (``idx < 0``) unchanged; the addition wraps in 64-bit two's complement.
    """
    idx = np.asarray(idx)
    if idx.ndim != 2:
        raise ValueError("idx must be [rows, topk]")
    rows = idx.shape[0]
    if sq <= 0 or rows % sq:
        raise ValueError("rows must be a multiple of sq")
    out = []
    for r in range(rows):
        off = (r // sq) * int(seqlen_kv)
        row = []
        for v in idx[r].tolist():
            w = v if v < 0 else v + off
            row.append((w + 2**63) % 2**64 - 2**63)   # exact Python ints, then wrap
        out.append(row)
    return np.array(out, dtype=np.int64).reshape(idx.shape)


def positions_batched(b: int, sq_per_batch: int, pos0: int = 0) -> np.ndarray:
    """Positions of ``b`` sequences of ``sq_per_batch`` tokens folded into one
    token axis (``B*S`` folding): row ``s`` sits at ``pos0 + s % sq_per_batch``."""
    s = np.arange(b * sq_per_batch, dtype=np.int64)
    return pos0 + s % sq_per_batch


def positions_contiguous(sq: int, pos0: int) -> np.ndarray:
    """Absolute positions ``pos0 .. pos0+sq-1`` of a contiguous shard."""
    return np.arange(pos0, pos0 + sq, dtype=np.int64)


__all__ = [
    "inv_freq", "rope_angles", "invrope", "rope", "postmix_fwd",
    "postmix_bwd", "postmix_bwd_dO", "postmix_bwd_dM", "postmix_fwd_grouped",
    "postmix_bwd_grouped", "postmix_bwd_grouped_dO", "kv_idx_local_to_global",
    "kv_idx_local_to_global_i64", "positions_contiguous", "positions_batched",
]
