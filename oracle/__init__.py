"""fp64 CPU oracle for the fused inverse-RoPE + VHA postmix and the KV index remap.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it. It shares no code with the
CUDA library (``partial_inverse_rope_gb300``) and imports nothing from it.
"""

from .invrope_oracle import (  # noqa: F401
    inv_freq,
    rope_angles,
    invrope,
    rope,
    postmix_fwd,
    postmix_bwd,
    postmix_bwd_dO,
    postmix_bwd_dM,
    postmix_fwd_grouped,
    postmix_bwd_grouped,
    postmix_bwd_grouped_dO,
    kv_idx_local_to_global,
    kv_idx_local_to_global_i64,
    positions_contiguous,
    positions_batched,
)
