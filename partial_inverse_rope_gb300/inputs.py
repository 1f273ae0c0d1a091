"""Seeded synthetic inputs for the postmix and remap workloads.

This module only draws random tensors of the workloads' shapes; it holds none
of the method's arithmetic, so both the CUDA path and the fp64 oracle can be
fed from it. Recipes (shapes from the production shard described in PaddleFleet
PR #1772, "Fuse HCA inverse RoPE into the VHA postmix, and the sparse-attention
KV index remap", English description item 1 and its measurement paragraph):

* ``O`` and ``dY``: N(0, 1) drawn in fp32 and rounded (RNE) to bf16,
  ``[sq, nh, nope+pe]``;
* ``M`` of layer ``l``: ``I + 0.02 * N(0, 1)`` in fp32, ``[nh, nh]``;
* KV index table: int32 ``[b*sq, topk]`` uniform in ``[0, seqlen_kv)`` with a
  fraction ``pad_frac`` of the entries replaced by ``-1`` padding.

Every tensor has its own generator: ``O`` uses ``seed``, ``dY`` ``seed+1`` and
the ``M`` of layer ``l`` ``seed+2+l``.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class PostmixConfig:
    name: str
    sq: int
    nh: int
    nope: int
    pe: int
    pos0: int
    theta: float = 10000.0
    seed: int = 0
    layers: int = 1

    @property
    def d(self) -> int:
        return self.nope + self.pe

    def fwd_bytes(self) -> int:
        """Algorithmic HBM bytes of one forward: read O, write Y (bf16), read M (fp32)."""
        return 2 * self.sq * self.nh * self.d * 2 + 4 * self.nh * self.nh

    def bwd_bytes(self) -> int:
        """Read dY and O, write dO (bf16); read M and write dM (fp32)."""
        return 3 * self.sq * self.nh * self.d * 2 + 8 * self.nh * self.nh


@dataclass(frozen=True)
class RemapConfig:
    name: str
    b: int
    sq: int
    topk: int
    seqlen_kv: int
    pad_frac: float = 0.05
    seed: int = 0

    @property
    def rows(self) -> int:
        return self.b * self.sq

    def bytes(self) -> int:
        """Read the int32 table once and write it once."""
        return 2 * self.rows * self.topk * 4


TINY = PostmixConfig("tiny", sq=128, nh=4, nope=48, pe=16, pos0=0)
MID = PostmixConfig("mid", sq=2048, nh=16, nope=448, pe=64, pos0=0)
PROD = PostmixConfig("production_shard", sq=16384, nh=64, nope=448, pe=64,
                     pos0=16384, layers=37)
SWEEP_NH3 = PostmixConfig("sweep_nh3", sq=8192, nh=3, nope=448, pe=64, pos0=0)
SWEEP_NH128 = PostmixConfig("sweep_nh128", sq=8192, nh=128, nope=448, pe=64, pos0=0)
POSTMIX_CONFIGS = {c.name: c for c in (TINY, MID, PROD, SWEEP_NH3, SWEEP_NH128)}

REMAP = RemapConfig("kv_remap", b=4, sq=16384, topk=2048, seqlen_kv=16384)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, seed: int, device="cpu") -> torch.Tensor:
    """N(0, 1) in fp32, rounded to nearest-even bf16."""
    g = _gen(seed, device)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    return x.to(torch.bfloat16)


def postmix_M(nh: int, seed: int, device="cpu") -> torch.Tensor:
    """``I + 0.02 * N(0, 1)`` in fp32."""
    g = _gen(seed, device)
    z = torch.randn(nh, nh, generator=g, device=device, dtype=torch.float32)
    return torch.eye(nh, device=device, dtype=torch.float32) + 0.02 * z


def postmix_Mg(ng: int, gs: int, seed: int, device="cpu") -> torch.Tensor:
    """Grouped mix ``[ng, gs, gs]``: ``I + 0.02 * N(0, 1)`` per group, fp32."""
    g = _gen(seed, device)
    z = torch.randn(ng, gs, gs, generator=g, device=device, dtype=torch.float32)
    return torch.eye(gs, device=device, dtype=torch.float32)[None] + 0.02 * z


def random_positions(sq: int, seed: int, low: int, high: int, device="cpu") -> torch.Tensor:
    """int32 ``[sq]`` positions drawn uniformly from ``[low, high)``."""
    g = _gen(seed, device)
    return torch.randint(low, high, (sq,), generator=g, device=device, dtype=torch.int32)


def postmix_inputs(cfg: PostmixConfig, device="cpu", layer: int = 0):
    """``(O, dY, M)`` for one layer of ``cfg``."""
    shape = (cfg.sq, cfg.nh, cfg.d)
    O = normal_bf16(shape, cfg.seed, device)
    dY = normal_bf16(shape, cfg.seed + 1, device)
    M = postmix_M(cfg.nh, cfg.seed + 2 + layer, device)
    return O, dY, M


def kv_index_table(cfg: RemapConfig, device="cpu") -> torch.Tensor:
    """int32 ``[b*sq, topk]`` uniform in ``[0, seqlen_kv)`` with ``-1`` padding."""
    g = _gen(cfg.seed, device)
    idx = torch.randint(0, cfg.seqlen_kv, (cfg.rows, cfg.topk), generator=g,
                        device=device, dtype=torch.int32)
    pad = torch.rand(cfg.rows, cfg.topk, generator=g, device=device) < cfg.pad_frac
    return torch.where(pad, torch.full_like(idx, -1), idx)


def positions(cfg: PostmixConfig) -> torch.Tensor:
    """Absolute positions ``pos0 .. pos0+sq-1`` of the shard (int64)."""
    return torch.arange(cfg.pos0, cfg.pos0 + cfg.sq, dtype=torch.int64)
