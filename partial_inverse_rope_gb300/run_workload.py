"""Run the library's kernels on a seeded synthetic workload (for profiling).

    python -m partial_inverse_rope_gb300.run_workload --ops fwd,bwd --sq 4096 --nh 64 --reps 2
    python -m partial_inverse_rope_gb300.run_workload --config sweep_nh128 --ops fwd,bwd --time

Each repetition calls the listed operations once, in the order given, on the
same resident inputs; the process exits non-zero if a kernel's watchdog fired.
Used to capture ncu profiles of one kernel on a case small enough to replay.
With --time, each call is timed with CUDA events on its stream (after 3
untimed repetitions; a 512 MiB buffer is rewritten between timed calls so that
inputs smaller than the L2 are not served from it) and the median per call is
printed with the algorithmic GB/s. With --host-cost N, each operation is
enqueued N times back to back through the C ABI (arguments marshalled once,
no synchronisation in between) and the host wall time per call is printed.
"""

from __future__ import annotations

import argparse
import sys

import torch

from . import binding as ir
from . import inputs as W


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--ops", default="fwd,bwd", help="comma list of fwd, bwd, remap")
    ap.add_argument("--sq", type=int, default=4096)
    ap.add_argument("--nh", type=int, default=64)
    ap.add_argument("--nope", type=int, default=448)
    ap.add_argument("--pe", type=int, default=64)
    ap.add_argument("--pos0", type=int, default=16384)
    ap.add_argument("--remap-rows", type=int, default=16384, help="rows of the remap table (b*sq)")
    ap.add_argument("--reps", type=int, default=2)
    ap.add_argument("--config", choices=sorted(W.POSTMIX_CONFIGS), default=None,
                    help="take sq/nh/nope/pe/pos0 from a named config")
    ap.add_argument("--time", action="store_true", help="time each call (median over --reps)")
    ap.add_argument("--host-cost", type=int, default=0, metavar="N",
                    help="host wall time per call over N back-to-back enqueues (keep N <= ~300: "
                         "the launches must fit the stream's queue, or the host waits for the GPU)")
    args = ap.parse_args(argv)

    ops = [o.strip() for o in args.ops.split(",") if o.strip()]
    dev = torch.device("cuda", 0)
    if args.config:
        c = W.POSTMIX_CONFIGS[args.config]
    else:
        c = W.PostmixConfig("workload", sq=args.sq, nh=args.nh, nope=args.nope, pe=args.pe, pos0=args.pos0)
    O, dY, M = W.postmix_inputs(c, device=dev)
    Y, dO = torch.empty_like(O), torch.empty_like(O)
    dM = torch.empty(c.nh, c.nh, dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, ir.invrope_postmix_bwd_workspace_bytes(c.sq, c.nh, c.nope, c.pe)),
                     dtype=torch.uint8, device=dev)
    R = W.RemapConfig("workload", b=max(1, args.remap_rows // 16384), sq=min(16384, args.remap_rows),
                      topk=2048, seqlen_kv=16384)
    idx = W.kv_index_table(R, device=dev) if "remap" in ops else None
    out = torch.empty_like(idx) if idx is not None else None
    def call(op):
        if op == "fwd":
            ir.invrope_postmix_fwd(O, M, c.pos0, c.nope, c.pe, c.theta, Y=Y)
        elif op == "bwd":
            ir.invrope_postmix_bwd(dY, O, M, c.pos0, c.nope, c.pe, c.theta, dO=dO, dM=dM, workspace=ws)
        elif op == "remap":
            ir.kv_idx_local_to_global(idx, R.sq, R.seqlen_kv, out=out)
        else:
            raise SystemExit(f"unknown op {op}")

    if args.host_cost:
        host_cost(ops, c, O, dY, M, Y, dO, dM, ws, R, idx, out, args.host_cost)
    elif not args.time:
        for _ in range(args.reps):
            for op in ops:
                call(op)
        torch.cuda.synchronize()
    else:
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        nbytes = {"fwd": c.fwd_bytes(), "bwd": c.bwd_bytes(), "remap": R.bytes()}
        for op in ops:
            for _ in range(3):
                call(op)
            times = []
            for _ in range(max(1, args.reps)):
                flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                call(op)
                e1.record()
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1) * 1e3)
            us = sorted(times)[len(times) // 2]
            print(f"{c.name} {op}: sq={c.sq} nh={c.nh} d={c.d} median {us:.2f} us over {len(times)} calls, "
                  f"{nbytes[op] / (us * 1e-6) / 1e9:.1f} GB/s algorithmic")
    fault = ir.invrope_take_device_fault()
    print(f"ran {args.reps} x {ops} at sq={c.sq} nh={c.nh} d={c.d}; watchdog fault code {fault}")
    return 1 if fault else 0


def host_cost(ops, c, O, dY, M, Y, dO, dM, ws, R, idx, out, n):
    """Host wall time per call of each op: the C-ABI entry point called n
    times with pre-marshalled ctypes arguments, without synchronising."""
    import ctypes
    import time

    lib = ir.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ws_bytes = ws.numel()
    argsets = {
        "fwd": (lib.invrope_postmix_fwd, (O.data_ptr(), M.data_ptr(), Y.data_ptr(), c.sq, c.nh, c.nope, c.pe,
                                          c.pos0, c.theta, stream)),
        "bwd": (lib.invrope_postmix_bwd, (dY.data_ptr(), O.data_ptr(), M.data_ptr(), dO.data_ptr(), dM.data_ptr(),
                                          ws.data_ptr(), ws_bytes, c.sq, c.nh, c.nope, c.pe, c.pos0, c.theta,
                                          stream)),
    }
    if idx is not None:
        argsets["remap"] = (lib.kv_idx_local_to_global, (idx.data_ptr(), out.data_ptr(), idx.shape[0],
                                                         idx.shape[1], R.sq, R.seqlen_kv, stream))
    # the same calls with an argument the library rejects first thing (sq or
    # rows < 0): the ctypes marshalling of these argument lists alone
    rejects = {
        "fwd": (-1,) + argsets["fwd"][1][4:],
        "bwd": (-1,) + argsets["bwd"][1][8:],
    }
    rejects["fwd"] = argsets["fwd"][1][:3] + rejects["fwd"]
    rejects["bwd"] = argsets["bwd"][1][:7] + rejects["bwd"]
    if idx is not None:
        rejects["remap"] = argsets["remap"][1][:2] + (-1,) + argsets["remap"][1][3:]
    for op in ops:
        fn, a = argsets[op]
        for _ in range(10):
            assert fn(*a) == 0
        torch.cuda.synchronize()
        # the GPU is held busy (a sleep kernel longer than the enqueue loop) so
        # that the calls queue up behind it: the loop then measures host time,
        # not the rate at which the GPU retires the launches
        torch.cuda._sleep(int(2e9 * 20e-6 * n))
        t0 = time.perf_counter()
        for _ in range(n):
            fn(*a)
        t1 = time.perf_counter()
        torch.cuda.synchronize()
        # the same argument list rejected at once: ctypes marshalling + the
        # first argument check, so the library's own host time is the difference
        ra = rejects[op]
        assert fn(*ra) != 0
        t2 = time.perf_counter()
        for _ in range(n):
            fn(*ra)
        t3 = time.perf_counter()
        full, marshal = 1e6 * (t1 - t0) / n, 1e6 * (t3 - t2) / n
        print(f"{c.name} {op}: host {full:.2f} us per call over {n} enqueues through ctypes; "
              f"the same call rejected at its first check {marshal:.2f} us; library {full - marshal:.2f} us")


if __name__ == "__main__":
    sys.exit(main())
