"""Run the library's kernels on a seeded synthetic workload (for profiling).

    python -m partial_inverse_rope_gb300.run_workload --ops fwd,bwd --sq 4096 --nh 64 --reps 2

Each repetition calls the listed operations once, in the order given, on the
same resident inputs; the process exits non-zero if a kernel's watchdog fired.
Used to capture ncu profiles of one kernel on a case small enough to replay.
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
    args = ap.parse_args(argv)

    ops = [o.strip() for o in args.ops.split(",") if o.strip()]
    dev = torch.device("cuda", 0)
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
    for _ in range(args.reps):
        for op in ops:
            if op == "fwd":
                ir.invrope_postmix_fwd(O, M, c.pos0, c.nope, c.pe, c.theta, Y=Y)
            elif op == "bwd":
                ir.invrope_postmix_bwd(dY, O, M, c.pos0, c.nope, c.pe, c.theta, dO=dO, dM=dM, workspace=ws)
            elif op == "remap":
                ir.kv_idx_local_to_global(idx, R.sq, R.seqlen_kv, out=out)
            else:
                raise SystemExit(f"unknown op {op}")
    torch.cuda.synchronize()
    fault = ir.invrope_take_device_fault()
    print(f"ran {args.reps} x {ops} at sq={c.sq} nh={c.nh} d={c.d}; watchdog fault code {fault}")
    return 1 if fault else 0


if __name__ == "__main__":
    sys.exit(main())
