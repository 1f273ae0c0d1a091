"""ctypes binding of ``libinvrope.so`` (the C ABI declared in ``include/invrope.h``).

Argument marshalling only: each function checks that torch tensors have the
dtype / device / layout the C ABI expects, allocates outputs with torch when
the caller passes none, and forwards raw device pointers, sizes and the
current CUDA stream. All arithmetic runs in the library's kernels. There is no
fallback: if the library is not built, the first call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

# INVROPE_LIBRARY selects another build of the same library (e.g. the
# debug-bounds build, libinvrope_debug.so); it must export the same symbols.
_LIB_PATH = os.environ.get("INVROPE_LIBRARY") or os.path.join(os.path.dirname(os.path.abspath(__file__)),
                                                             "libinvrope.so")
_lib = None

INVROPE_OK = 0
INVROPE_ERR_INVALID_ARG = 1
INVROPE_ERR_UNSUPPORTED = 2
INVROPE_ERR_WORKSPACE = 3
INVROPE_ERR_CUDA = 4
INVROPE_ERR_DEVICE = 5

# name -> (restype, argtypes); mirrors include/invrope.h
_SIGNATURES = {
    "invrope_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "invrope_last_cuda_error": (ctypes.c_int, []),
    "invrope_postmix_fwd": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int64, ctypes.c_double, ctypes.c_void_p]),
    "invrope_postmix_bwd_workspace_bytes": (ctypes.c_size_t, [
        ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "invrope_postmix_bwd": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_size_t,
        ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int64, ctypes.c_double, ctypes.c_void_p]),
    "invrope_postmix_bwd_noalloc": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int64, ctypes.c_double, ctypes.c_void_p]),
    "invrope_postmix_fwd_ex": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p]),
    "invrope_postmix_bwd_ex": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_void_p, ctypes.c_size_t,
        ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p]),
    "kv_idx_local_to_global": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]),
    "kv_idx_local_to_global_i64": (ctypes.c_int, [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]),
    "invrope_take_device_fault": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int)]),
    "invrope_watchdog_selftest": (ctypes.c_int, [ctypes.c_int64, ctypes.POINTER(ctypes.c_int)]),
    "invrope_debug_occupy_next_slot": (ctypes.c_int, [ctypes.c_int, ctypes.c_ulonglong]),
}

INVROPE_WATCHDOG_SELFTEST_CODE = 0x60A
INVROPE_FAULT_SCHED_BUSY_FWD = 0x5C1
INVROPE_FAULT_SCHED_BUSY_REMAP = 0x5C2
INVROPE_FAULT_SCHED_BUSY_BWD = 0x5C3


class InvropeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = lib().invrope_status_string(status).decode()
        if status == INVROPE_ERR_CUDA:
            msg += f" (cudaError {lib().invrope_last_cuda_error()})"
        super().__init__(f"{what}: {msg}")


def lib_path() -> str:
    return _LIB_PATH


def lib():
    """Load ``libinvrope.so`` once; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(
                f"{_LIB_PATH} is missing: build it with "
                "`python -m partial_inverse_rope_gb300.build` (there is no CPU fallback)")
        handle = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(status: int, what: str):
    if status != INVROPE_OK:
        raise InvropeError(status, what)


def _stream_handle(device, stream):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t, name, dtype, ndim):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def invrope_postmix_fwd(O, M, pos0: int, nope: int, pe: int, theta: float = 10000.0,
                        Y=None, stream=None):
    """``Y[s,g,:] = sum_h M[g,h] invrope_{pos0+s}(O[s,h,:])``; returns ``Y`` (bf16)."""
    _need(O, "O", torch.bfloat16, 3)
    _need(M, "M", torch.float32, 2)
    sq, nh, d = O.shape
    if tuple(M.shape) != (nh, nh):
        raise ValueError(f"M must be [{nh}, {nh}]")
    if Y is None:
        Y = torch.empty_like(O)
    else:
        _need(Y, "Y", torch.bfloat16, 3)
        if Y.shape != O.shape:
            raise ValueError("Y must have O's shape")
    st = lib().invrope_postmix_fwd(O.data_ptr(), M.data_ptr(), Y.data_ptr(), sq, nh, nope, pe,
                                   int(pos0), float(theta), _stream_handle(O.device, stream))
    _check(st, "invrope_postmix_fwd")
    return Y


def invrope_postmix_bwd_workspace_bytes(sq: int, nh: int, nope: int, pe: int) -> int:
    """Workspace bytes the backward needs on the current device (0 if the shape is invalid)."""
    return int(lib().invrope_postmix_bwd_workspace_bytes(int(sq), int(nh), int(nope), int(pe)))


def invrope_postmix_bwd(dY, O, M, pos0: int, nope: int, pe: int, theta: float = 10000.0,
                        dO=None, dM=None, workspace=None, stream=None):
    """Backward of the fused postmix; returns ``(dO bf16, dM fp32)``."""
    _need(dY, "dY", torch.bfloat16, 3)
    _need(O, "O", torch.bfloat16, 3)
    _need(M, "M", torch.float32, 2)
    sq, nh, d = O.shape
    if dY.shape != O.shape or tuple(M.shape) != (nh, nh):
        raise ValueError("dY must match O and M must be [nh, nh]")
    if dO is None:
        dO = torch.empty_like(O)
    if dM is None:
        dM = torch.empty(nh, nh, dtype=torch.float32, device=O.device)
    _need(dO, "dO", torch.bfloat16, 3)
    _need(dM, "dM", torch.float32, 2)
    if workspace is None:
        nbytes = invrope_postmix_bwd_workspace_bytes(sq, nh, nope, pe)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=O.device)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().invrope_postmix_bwd(dY.data_ptr(), O.data_ptr(), M.data_ptr(), dO.data_ptr(),
                                   dM.data_ptr(), workspace.data_ptr(), ws_bytes, sq, nh, nope, pe,
                                   int(pos0), float(theta), _stream_handle(O.device, stream))
    _check(st, "invrope_postmix_bwd")
    return dO, dM


def _mix_and_positions(M, positions, sq, nh, group_size, device):
    """Check the [nh/gs, gs, gs] mix and the optional int32 [sq] positions."""
    gs = nh if group_size is None else int(group_size)
    if gs < 1 or nh % gs:
        raise ValueError("group_size must divide nh")
    want = (nh // gs, gs, gs) if group_size is not None else (nh, nh)
    _need(M, "M", torch.float32, len(want))
    if tuple(M.shape) != want:
        raise ValueError(f"M must be {list(want)}")
    if positions is not None:
        _need(positions, "positions", torch.int32, 1)
        if positions.shape[0] != sq or positions.device != device:
            raise ValueError("positions must be int32 [sq] on the tensors' device")
    return gs, (positions.data_ptr() if positions is not None else None)


def invrope_postmix_fwd_ex(O, M, nope: int, pe: int, positions=None, pos0: int = 0,
                           theta: float = 10000.0, group_size=None, Y=None, stream=None):
    """Forward with an optional grouped mix (``M`` = [nh/gs, gs, gs] when
    ``group_size`` is given) and optional int32 per-row ``positions`` (row s
    sits at ``pos0 + positions[s]``, else ``pos0 + s``); returns ``Y``."""
    _need(O, "O", torch.bfloat16, 3)
    sq, nh, d = O.shape
    gs, pos_ptr = _mix_and_positions(M, positions, sq, nh, group_size, O.device)
    if Y is None:
        Y = torch.empty_like(O)
    else:
        _need(Y, "Y", torch.bfloat16, 3)
        if Y.shape != O.shape:
            raise ValueError("Y must have O's shape")
    st = lib().invrope_postmix_fwd_ex(O.data_ptr(), M.data_ptr(), Y.data_ptr(), sq, nh, gs, nope, pe,
                                      pos_ptr, int(pos0), float(theta), _stream_handle(O.device, stream))
    _check(st, "invrope_postmix_fwd_ex")
    return Y


def invrope_postmix_bwd_ex(dY, O, M, nope: int, pe: int, positions=None, pos0: int = 0,
                           theta: float = 10000.0, group_size=None, dO=None, dM=None,
                           workspace=None, stream=None):
    """Backward of :func:`invrope_postmix_fwd_ex`; returns ``(dO bf16, dM fp32)``
    with ``dM`` shaped like ``M``."""
    _need(dY, "dY", torch.bfloat16, 3)
    _need(O, "O", torch.bfloat16, 3)
    sq, nh, d = O.shape
    if dY.shape != O.shape:
        raise ValueError("dY must match O")
    gs, pos_ptr = _mix_and_positions(M, positions, sq, nh, group_size, O.device)
    if dO is None:
        dO = torch.empty_like(O)
    if dM is None:
        dM = torch.empty(M.shape, dtype=torch.float32, device=O.device)
    _need(dO, "dO", torch.bfloat16, 3)
    _need(dM, "dM", torch.float32, M.dim())
    if dM.shape != M.shape:
        raise ValueError("dM must have M's shape")
    if workspace is None:
        nbytes = invrope_postmix_bwd_workspace_bytes(sq, nh, nope, pe)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=O.device)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib().invrope_postmix_bwd_ex(dY.data_ptr(), O.data_ptr(), M.data_ptr(), dO.data_ptr(),
                                      dM.data_ptr(), workspace.data_ptr(), ws_bytes, sq, nh, gs, nope, pe,
                                      pos_ptr, int(pos0), float(theta), _stream_handle(O.device, stream))
    _check(st, "invrope_postmix_bwd_ex")
    return dO, dM


def invrope_postmix_bwd_noalloc(dY, O, M, pos0: int, nope: int, pe: int, dO, dM,
                                theta: float = 10000.0, stream=None):
    """Backward without a workspace, for callers that may not allocate device
    memory on their call path: the library's own fixed scratch array
    (``INVROPE_NOALLOC_SCRATCH_BYTES``) holds the dM partials. ``dO`` and
    ``dM`` must be given (this wrapper allocates nothing either). Calls that
    overlap on the GPU share that array and must be ordered."""
    _need(dY, "dY", torch.bfloat16, 3)
    _need(O, "O", torch.bfloat16, 3)
    _need(M, "M", torch.float32, 2)
    _need(dO, "dO", torch.bfloat16, 3)
    _need(dM, "dM", torch.float32, 2)
    sq, nh, d = O.shape
    if dY.shape != O.shape or dO.shape != O.shape or tuple(M.shape) != (nh, nh) \
            or tuple(dM.shape) != (nh, nh):
        raise ValueError("dY/dO must match O; M and dM must be [nh, nh]")
    st = lib().invrope_postmix_bwd_noalloc(dY.data_ptr(), O.data_ptr(), M.data_ptr(), dO.data_ptr(),
                                           dM.data_ptr(), sq, nh, nope, pe, int(pos0), float(theta),
                                           _stream_handle(O.device, stream))
    _check(st, "invrope_postmix_bwd_noalloc")
    return dO, dM


def kv_idx_local_to_global(idx, sq: int, seqlen_kv: int, out=None, stream=None):
    """``out = idx < 0 ? idx : idx + (row // sq) * seqlen_kv`` on an int32 ``[rows, topk]`` table."""
    _need(idx, "idx", torch.int32, 2)
    rows, topk = idx.shape
    if out is None:
        out = torch.empty_like(idx)
    else:
        _need(out, "out", torch.int32, 2)
        if out.shape != idx.shape:
            raise ValueError("out must match idx")
    st = lib().kv_idx_local_to_global(idx.data_ptr(), out.data_ptr(), rows, topk, int(sq),
                                      int(seqlen_kv), _stream_handle(idx.device, stream))
    _check(st, "kv_idx_local_to_global")
    return out


def kv_idx_local_to_global_i64(idx, sq: int, seqlen_kv: int, out=None, stream=None):
    """The same remap on an int64 ``[rows, topk]`` table (64-bit wrap)."""
    _need(idx, "idx", torch.int64, 2)
    rows, topk = idx.shape
    if out is None:
        out = torch.empty_like(idx)
    else:
        _need(out, "out", torch.int64, 2)
        if out.shape != idx.shape:
            raise ValueError("out must match idx")
    st = lib().kv_idx_local_to_global_i64(idx.data_ptr(), out.data_ptr(), rows, topk, int(sq),
                                          int(seqlen_kv), _stream_handle(idx.device, stream))
    _check(st, "kv_idx_local_to_global_i64")
    return out


def invrope_take_device_fault() -> int:
    """Synchronise, then return and clear the kernels' watchdog code (0 = no fault)."""
    v = ctypes.c_int(0)
    _check(lib().invrope_take_device_fault(ctypes.byref(v)), "invrope_take_device_fault")
    return v.value


def invrope_debug_occupy_next_slot(which: str, owner: int) -> None:
    """Test hook: mark the work-counter slot the next eager ``"fwd"`` or
    ``"remap"`` launch will take as held by launch tag ``owner``."""
    code = {"fwd": 0, "remap": 1}[which]
    _check(lib().invrope_debug_occupy_next_slot(code, int(owner)), "invrope_debug_occupy_next_slot")


def invrope_watchdog_selftest(limit_us: int = 50000) -> int:
    """Run one bounded wait that must expire; returns the recorded watchdog code."""
    v = ctypes.c_int(0)
    _check(lib().invrope_watchdog_selftest(int(limit_us), ctypes.byref(v)), "invrope_watchdog_selftest")
    return v.value
