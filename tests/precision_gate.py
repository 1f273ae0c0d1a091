"""A gate for "the rotation is applied in fp32 to unrounded values and the
result is rounded to bf16 once", the reading of ``high_precision_rope=True``
(PaddleFleet PR #1772, Chinese description section 1, and PR #1843 item 1 list
it among the settings the fused path hands back; neither page defines it).

For a rotated output y = x1 cos a - x2 sin a (or its partner) with exact value
``exact`` (fp64 oracle), a kernel that forms y in fp32 with an error of at most
eps and then rounds once to nearest-even bf16 returns Y with

    |Y - exact| <= 0.5 ulp(exact) + 2 eps

(Y is at least as close to the fp32 value as the bf16 neighbour R of
``exact`` is, and |R - exact| <= 0.5 ulp(exact)). The fp32 error is bounded
by the magnitude of the terms: ``scale`` = sum over the mixed heads of
|M| (|x1| + |x2|) for the pair.

* head mix with M carried as bf16 hi + lo: |M - hi - lo| <= 2^-17 |M|, and
  fp32 accumulation of 2 nh <= 256 products: <= 2^-16 scale in all;
* angle reduced exactly to 2^-32 turns, then fp32: <= ~4e-7 rad; sin/cos to
  2^-21.4; two products and a sum in fp32: together <= 2^-20 scale.

So eps <= 2^-15.9 scale, and the gate allows 0.5 ulp(exact) + 2^-14 scale.
A rotation that touches a bf16-rounded value (the mixed result rounded before
it is rotated, bf16 sine / cosine, bf16 products, or the inputs rotated and
rounded before the mix) adds an error of about 2^-9 of the value and puts a
large share of the outputs outside the gate; ``tests/test_precision_gate.py``
shows that on emulated kernels of each kind.
"""

from __future__ import annotations

import numpy as np

GATE_EPS = 2.0 ** -14


def ulp_bf16(v) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significand bits; subnormal spacing
    2^-133 below 2^-126)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def rne_bf16(v) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value, ties to even, in one step
    (no intermediate fp32 rounding)."""
    v = np.asarray(v, dtype=np.float64)
    u = ulp_bf16(v)
    return np.rint(v / u) * u  # v / u is exact (power of two); rint ties to even


def rotation_gate(got, exact, scale):
    """Return (mask of elements outside the gate, error in ulps of exact)."""
    got = np.asarray(got, dtype=np.float64)
    exact = np.asarray(exact, dtype=np.float64)
    err = np.abs(got - exact)
    allowed = 0.5 * ulp_bf16(exact) + GATE_EPS * np.asarray(scale, dtype=np.float64)
    return err > allowed, err / ulp_bf16(exact)


def pair_scale(x, M_abs_t, nope: int, pe: int) -> np.ndarray:
    """Per pe channel of every (s, head): sum_h |M|[., h] (|x1| + |x2|) of its
    pair, for x [sq, nh, d] and ``M_abs_t`` the transposed |mix| applied to
    the heads (|M|^T for the forward, |M| for the backward's M^T)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    h = pe // 2
    t = x[:, :, nope:nope + h] + x[:, :, nope + h:nope + pe]
    mixed = np.einsum("shi,hg->sgi", t, M_abs_t)
    return np.concatenate([mixed, mixed], axis=2)
