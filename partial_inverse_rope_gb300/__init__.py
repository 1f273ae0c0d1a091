"""GB300-native fused inverse RoPE + VHA postmix (forward / backward) and the
sparse-attention KV index remap, as hand-written sm_103a CUDA kernels behind a
C ABI (``include/invrope.h``), with a thin ctypes binding of the same names.
"""

from .binding import (  # noqa: F401
    InvropeError,
    invrope_debug_occupy_next_slot,
    invrope_postmix_bwd,
    invrope_postmix_bwd_ex,
    invrope_postmix_bwd_noalloc,
    invrope_postmix_bwd_workspace_bytes,
    invrope_postmix_fwd,
    invrope_postmix_fwd_ex,
    invrope_take_device_fault,
    invrope_watchdog_selftest,
    kv_idx_local_to_global,
    kv_idx_local_to_global_i64,
    lib,
    lib_path,
)
