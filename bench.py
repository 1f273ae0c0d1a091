"""Benchmark of the fused inverse-RoPE + VHA postmix hot path on GB300.

One step = one layer of the production shard: forward (Y), backward (dO, dM)
and one KV index remap of the remap workload. The timed region runs K steps
back to back with a fresh M per layer (37 layers cycled), inputs resident in
HBM (1 GiB O / dY and a 512 MiB index table, each larger than the 129 MB L2, so
no flush is needed between steps). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle (the only reference this
method has here) on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from partial_inverse_rope_gb300 import inputs as W  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["partial_inverse_rope_gb300/csrc/postmix.cu",
                  "partial_inverse_rope_gb300/csrc/ptx.cuh",
                  "partial_inverse_rope_gb300/csrc/sched.cuh"]
# machine-readable ncu counters of the backward kernel (written beside its summary)
PROFILE_COUNTERS = os.path.join(ROOT, "profiles", "postmix_bwd_production_shard.json")


# ---------------------------------------------------------------- environment
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """Per-launch DRAM bytes of the backward kernel from the committed ncu
    counters (JSON), or None when they are missing or were taken with another
    kernel source."""
    try:
        with open(PROFILE_COUNTERS) as f:
            rec = json.load(f)
        if rec["kernel_source_sha256_16"] != kernel_source_hash():
            return None
        return int(rec["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError, TypeError):
        return None


class ClockSampler:
    """nvidia-smi samples (every 25 ms: a short timed region still gets a few)
    taken while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []  # (host time, csv line)
        self.thread = None
        self.t_start = None
        self.t_stop = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark_start(self):
        self.t_start = time.perf_counter()

    def mark_stop(self):
        self.t_stop = time.perf_counter()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        window = [ln for t, ln in self.lines
                  if self.t_start is None or self.t_start <= t <= (self.t_stop or t)]
        for line in window:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world, local):
    import partial_inverse_rope_gb300 as ir

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    c = W.PROD
    R = W.REMAP
    # inputs resident in HBM (seeded, synthetic)
    O, dY, _ = W.postmix_inputs(c, device=dev)
    Ms = [W.postmix_M(c.nh, c.seed + 2 + l, dev) for l in range(c.layers)]
    idx = W.kv_index_table(R, device=dev)
    Y = torch.empty_like(O)
    dO = torch.empty_like(O)
    dM = torch.empty(c.nh, c.nh, dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, ir.invrope_postmix_bwd_workspace_bytes(c.sq, c.nh, c.nope, c.pe)),
                     dtype=torch.uint8, device=dev)
    out = torch.empty_like(idx)
    stream = torch.cuda.current_stream(dev)

    def step(l, ev=None):
        M = Ms[l % len(Ms)]
        if ev is not None:
            ev[0].record(stream)
        ir.invrope_postmix_fwd(O, M, c.pos0, c.nope, c.pe, c.theta, Y=Y)
        if ev is not None:
            ev[1].record(stream)
        ir.invrope_postmix_bwd(dY, O, M, c.pos0, c.nope, c.pe, c.theta, dO=dO, dM=dM, workspace=ws)
        if ev is not None:
            ev[2].record(stream)
        ir.kv_idx_local_to_global(idx, R.sq, R.seqlen_kv, out=out)
        if ev is not None:
            ev[3].record(stream)

    for l in range(args.warmup):
        step(l)
    torch.cuda.synchronize()

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        clocks.mark_start()
        t0.record(stream)
        for k in range(args.steps):
            step(k, events[k])
        t1.record(stream)
        torch.cuda.synchronize()
        clocks.mark_stop()
    barrier(world)
    ms_total = t0.elapsed_time(t1)
    fwd_us = [e[0].elapsed_time(e[1]) * 1e3 for e in events]
    bwd_us = [e[1].elapsed_time(e[2]) * 1e3 for e in events]
    remap_us = [e[2].elapsed_time(e[3]) * 1e3 for e in events]
    ms_total = max_over_ranks(ms_total, world)
    fault = ir.invrope_take_device_fault()

    step_bytes = c.fwd_bytes() + c.bwd_bytes() + R.bytes()
    ms_per_step = ms_total / args.steps
    value = whole_job_gbs(step_bytes, ms_per_step, world)  # GB/s over all ranks

    # end to end through the public API with host buffers: pinned host -> device
    # inputs, the three calls, device -> pinned host outputs, all inside the timed region
    e2e = run_e2e(args, ir, c, R, dev, stream, O, dY, Ms, idx, Y, dO, dM, ws, out, world)

    peak, peak_kind = measured_peak()
    configs = config_sweep(ir, dev, stream, peak) if rank == 0 else None
    bwd_avg = statistics.mean(bwd_us)
    achieved = c.bwd_bytes() / (bwd_avg * 1e-6) / 1e9
    line = {
        "metric": "fused inv-RoPE+postmix fwd/bwd us and HBM GB/s (% of roof), sq=16384 nh=64",
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) bf16 O/dY, M = I + 0.02 N(0,1) fp32 per layer, "
                "int32 uniform KV table with 5% -1 padding",
        "config": {
            "workload": "production shard fwd+bwd (sq=16384, nh=64, nope=448, pe=64, positions "
                        "16384..32767, 37 layers cycled) + KV index remap (b=4, sq=16384, "
                        "topk=2048, seqlen_kv=16384)",
            "sq": c.sq, "nh": c.nh, "nope": c.nope, "pe": c.pe, "pos0": c.pos0,
            "theta": c.theta, "layers": c.layers,
            "remap": {"b": R.b, "sq": R.sq, "topk": R.topk, "seqlen_kv": R.seqlen_kv},
            "parallelism": "replicas" if world > 1 else "single",
            "l2": "inputs larger than L2 (1 GiB / 512 MiB per tensor), no flush",
        },
        "kernels_us": {
            "fwd": round(statistics.mean(fwd_us), 2),
            "bwd": round(bwd_avg, 2),
            "remap": round(statistics.mean(remap_us), 2),
        },
        "kernels_gbs": {
            "fwd": round(c.fwd_bytes() / (statistics.mean(fwd_us) * 1e-6) / 1e9, 1),
            "bwd": round(achieved, 1),
            "remap": round(R.bytes() / (statistics.mean(remap_us) * 1e-6) / 1e9, 1),
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "invrope_postmix_bwd (main kernel + dM reduce, per call)",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic(),
            "algorithmic_bytes_per_launch": c.bwd_bytes(),
        },
        "e2e": e2e,
        "gpu_launches": args.steps * 4,
        "clocks": clocks.summary(),
        "device_fault": fault,
    }
    if rank == 0:
        base = cpu_baseline(args)
        line["cpu_baseline"] = base
        # the production shard's oracle time per config line: the cpu_baseline run itself
        prod = configs[W.PROD.name]["oracle"]
        prod.update({"rows": base["rows"], "fwd_bwd_s": base["postmix_s"], "cores": base["cores"]})
        prod["gbs"] = round((W.PROD.fwd_bytes() + W.PROD.bwd_bytes()) * base["rows"] / W.PROD.sq
                            / base["postmix_s"] / 1e9, 3)
        line["configs"] = configs
        print(json.dumps(line), flush=True)


# rows of each config the oracle runs in the per-config sweep (the rest scale)
CONFIG_ORACLE_ROWS = {"tiny": 128, "mid": 2048, "sweep_nh3": 8192, "sweep_nh128": 2048}


def config_sweep(ir, dev, stream, peak):
    """Every postmix config: forward and backward timed alone with CUDA events
    (median of 20 calls, a 512 MiB buffer rewritten before each so that no
    input is served from the 129 MB L2), algorithmic GB/s and the fraction of
    the measured copy peak; beside it the fp64 oracle's time for fwd + bwd on
    the host cores (all rows, or a leading block of rows scaled to the config;
    the production shard's oracle time is the cpu_baseline run).

    A single call of a small config is bounded by fixed costs: the event pair
    around one trivial kernel already reads ~6 us on this GPU. For the configs
    whose inputs fit in the L2, `stream` adds the per-call device time of
    back-to-back calls: the calls are queued behind a sleep kernel (so the host
    enqueue time is not measured), rotate over enough input/output sets that a
    set comes back only after >= 256 MB (twice the L2) of the other sets'
    traffic (at most 64 sets: tiny stays L2-resident and says so), and one
    event pair spans them all."""
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    res = {}
    for c in (W.TINY, W.MID, W.SWEEP_NH3, W.SWEEP_NH128, W.PROD):
        O, dY, M = W.postmix_inputs(c, device=dev)
        Y, dO = torch.empty_like(O), torch.empty_like(O)
        dM = torch.empty(c.nh, c.nh, dtype=torch.float32, device=dev)
        ws = torch.empty(max(16, ir.invrope_postmix_bwd_workspace_bytes(c.sq, c.nh, c.nope, c.pe)),
                         dtype=torch.uint8, device=dev)
        calls = {
            "fwd": lambda: ir.invrope_postmix_fwd(O, M, c.pos0, c.nope, c.pe, c.theta, Y=Y),
            "bwd": lambda: ir.invrope_postmix_bwd(dY, O, M, c.pos0, c.nope, c.pe, c.theta, dO=dO, dM=dM,
                                                  workspace=ws),
        }
        nbytes = {"fwd": c.fwd_bytes(), "bwd": c.bwd_bytes()}
        row = {"shape": [c.sq, c.nh, c.nope, c.pe], "pos0": c.pos0}
        for name, fn in calls.items():
            for _ in range(3):
                fn()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
            for e0, e1 in ev:
                flush.fill_(1)
                e0.record(stream)
                fn()
                e1.record(stream)
            torch.cuda.synchronize()
            us = statistics.median(e0.elapsed_time(e1) * 1e3 for e0, e1 in ev)
            gbs = nbytes[name] / (us * 1e-6) / 1e9
            row[f"{name}_us"] = round(us, 2)
            row[f"{name}_gbs"] = round(gbs, 1)
            row[f"{name}_frac"] = round(gbs / peak, 4)
        if c.fwd_bytes() < (128 << 20):
            row["stream"] = stream_sweep(ir, dev, stream, c, peak)
        del O, dY, Y, dO, ws
        row["oracle"] = oracle_config(c) if c.name in CONFIG_ORACLE_ROWS else {"kind": "oracle"}
        res[c.name] = row
    del flush
    torch.cuda.empty_cache()
    return res


def stream_sweep(ir, dev, stream, c, peak, calls_per_rep=64):
    """Per-call device time of back-to-back forward / backward calls of config
    `c` over rotating input sets (see config_sweep)."""
    set_bytes = {"fwd": c.fwd_bytes(), "bwd": c.bwd_bytes()}
    out = {}
    for name in ("fwd", "bwd"):
        nsets = min(64, 1 + -(-(256 << 20) // set_bytes[name]))
        sets = []
        for j in range(nsets):
            cj = W.PostmixConfig(c.name, sq=c.sq, nh=c.nh, nope=c.nope, pe=c.pe, pos0=c.pos0, seed=c.seed + j)
            O, dY, M = W.postmix_inputs(cj, device=dev)
            res = torch.empty_like(O)
            dM = torch.empty(c.nh, c.nh, dtype=torch.float32, device=dev)
            ws = torch.empty(max(16, ir.invrope_postmix_bwd_workspace_bytes(c.sq, c.nh, c.nope, c.pe)),
                             dtype=torch.uint8, device=dev) if name == "bwd" else None
            sets.append((O, dY, M, res, dM, ws))
        del O, dY, M, res, dM, ws

        def call(j):
            O, dY, M, res, dM, ws = sets[j % nsets]
            if name == "fwd":
                ir.invrope_postmix_fwd(O, M, c.pos0, c.nope, c.pe, c.theta, Y=res)
            else:
                ir.invrope_postmix_bwd(dY, O, M, c.pos0, c.nope, c.pe, c.theta, dO=res, dM=dM, workspace=ws)
        for j in range(nsets):
            call(j)
        per = []
        for _ in range(5):
            torch.cuda.synchronize()
            torch.cuda._sleep(int(2e9 * 30e-6 * calls_per_rep))  # covers the host's enqueue of the calls
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for j in range(calls_per_rep):
                call(j)
            e1.record(stream)
            torch.cuda.synchronize()
            per.append(e0.elapsed_time(e1) * 1e3 / calls_per_rep)
        us = statistics.median(per)
        gbs = set_bytes[name] / (us * 1e-6) / 1e9
        out[f"{name}_us"] = round(us, 2)
        out[f"{name}_gbs"] = round(gbs, 1)
        out[f"{name}_frac"] = round(gbs / peak, 4)
        out[f"{name}_sets"] = nsets
        del sets
    out["l2"] = ("inputs L2-resident (64 sets of the config fit in L2)" if 63 * c.fwd_bytes() < (256 << 20)
                 else "a set comes back after >= 256 MB of other sets' traffic")
    out["calls"] = calls_per_rep
    torch.cuda.empty_cache()
    return out


def oracle_config(c):
    """fp64 oracle fwd + bwd (dO, dM) on the first rows of config `c`."""
    import numpy as np

    import oracle

    rows = min(c.sq, CONFIG_ORACLE_ROWS[c.name])
    sub = W.PostmixConfig(c.name, sq=rows, nh=c.nh, nope=c.nope, pe=c.pe, pos0=c.pos0, seed=c.seed)
    O, dY, M = W.postmix_inputs(sub, device="cpu")
    O64, dY64, M64 = (t.to(torch.float64).numpy() for t in (O, dY, M))
    pos = np.arange(c.pos0, c.pos0 + rows, dtype=np.int64)
    t0 = time.perf_counter()
    oracle.postmix_fwd(O64, M64, pos, c.nope, c.pe, c.theta)
    oracle.postmix_bwd(dY64, O64, M64, pos, c.nope, c.pe, c.theta)
    dt = time.perf_counter() - t0
    return {"kind": "oracle", "rows": rows, "fwd_bwd_s": round(dt, 4), "cores": oracle_threads(),
            "gbs": round((c.fwd_bytes() + c.bwd_bytes()) * rows / c.sq / dt / 1e9, 3)}


def run_e2e(args, ir, c, R, dev, stream, O, dY, Ms, idx, Y, dO, dM, ws, out, world):
    """End to end through the public API with host buffers: every step copies
    its inputs (O, dY, M, the KV table) from pinned host memory to the device,
    runs the three calls, and copies its results (Y, dO, dM, the remapped
    table) back to pinned host memory, all inside the timed region. Steps are
    software-pipelined the way a caller streaming layers would run them: two
    device buffer sets and three streams, so step k+1's inputs go up and step
    k-1's results come down while step k computes."""
    nset = 2
    L = len(Ms)
    hO = torch.empty(O.shape, dtype=O.dtype, pin_memory=True)
    hdY = torch.empty(dY.shape, dtype=dY.dtype, pin_memory=True)
    hM = [torch.empty(m.shape, dtype=m.dtype, pin_memory=True) for m in Ms]
    hidx = torch.empty(idx.shape, dtype=idx.dtype, pin_memory=True)
    hO.copy_(O)
    hdY.copy_(dY)
    for h, m in zip(hM, Ms):
        h.copy_(m)
    hidx.copy_(idx)
    # device buffer sets (set 0 reuses the resident tensors)
    d_in = [(O, dY, torch.empty_like(Ms[0]), idx)] + [
        (torch.empty_like(O), torch.empty_like(dY), torch.empty_like(Ms[0]), torch.empty_like(idx))
        for _ in range(nset - 1)]
    d_out = [(Y, dO, dM, out)] + [
        (torch.empty_like(Y), torch.empty_like(dO), torch.empty_like(dM), torch.empty_like(out))
        for _ in range(nset - 1)]
    h_out = [tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in d_out[0])
             for _ in range(nset)]
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = {k: [torch.cuda.Event() for _ in range(nset)] for k in ("in", "comp", "out")}

    def e2e_step(k):
        b = k % nset
        Oi, dYi, Mi, idxi = d_in[b]
        Yo, dOo, dMo, outo = d_out[b]
        with torch.cuda.stream(s_in):
            if k >= nset:
                s_in.wait_event(ev["comp"][b])   # set b's inputs are free again
            Oi.copy_(hO, non_blocking=True)
            dYi.copy_(hdY, non_blocking=True)
            Mi.copy_(hM[k % L], non_blocking=True)
            idxi.copy_(hidx, non_blocking=True)
            ev["in"][b].record(s_in)
        s_comp.wait_event(ev["in"][b])
        if k >= nset:
            s_comp.wait_event(ev["out"][b])      # set b's results have been copied out
        ir.invrope_postmix_fwd(Oi, Mi, c.pos0, c.nope, c.pe, c.theta, Y=Yo, stream=s_comp)
        ir.invrope_postmix_bwd(dYi, Oi, Mi, c.pos0, c.nope, c.pe, c.theta, dO=dOo, dM=dMo, workspace=ws,
                               stream=s_comp)
        ir.kv_idx_local_to_global(idxi, R.sq, R.seqlen_kv, out=outo, stream=s_comp)
        ev["comp"][b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["comp"][b])
            for h, d in zip(h_out[b], d_out[b]):
                h.copy_(d, non_blocking=True)
            ev["out"][b].record(s_out)

    steps = max(1, min(args.steps, 12))
    for k in range(min(2, args.warmup)):
        e2e_step(k)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for k in range(steps):
        e2e_step(k)
    torch.cuda.synchronize()
    dt = max_over_ranks((time.perf_counter() - t0) * 1e3, world) / steps
    step_bytes = c.fwd_bytes() + c.bwd_bytes() + R.bytes()
    h2d = hO.numel() * 2 + hdY.numel() * 2 + c.nh * c.nh * 4 + hidx.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    return {"value": round(whole_job_gbs(step_bytes, dt, world), 1), "unit": "GB/s",
            "ms_per_step": round(dt, 3), "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelining": "2 buffer sets, 3 streams: copies of neighbouring steps overlap this step's compute"}


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Largest value of ``x`` over all ranks (the slowest replica's time)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(step_bytes, ms_per_step_max, world):
    """Weak-scaling aggregate: every replica moves ``step_bytes`` per step; the
    job's rate is all ranks' bytes over the slowest rank's time per step."""
    return world * step_bytes / (ms_per_step_max * 1e-3) / 1e9


# ---------------------------------------------------------------- oracle (CPU) legs
def oracle_sample(rows: int, threads_note=True):
    """Time the fp64 oracle on the first `rows` positions of the production shard
    (fwd + bwd incl. dM) plus a proportional slice of the remap table; returns
    (seconds, algorithmic bytes covered)."""
    import numpy as np

    import oracle

    c = W.PROD
    R = W.REMAP
    O, dY, M = W.postmix_inputs(W.PostmixConfig("sample", sq=rows, nh=c.nh, nope=c.nope, pe=c.pe,
                                                pos0=c.pos0, seed=c.seed), device="cpu")
    frac = rows / c.sq
    remap_rows = max(R.sq, int(R.rows * frac) // R.sq * R.sq)
    idx = W.kv_index_table(W.RemapConfig("sample", b=remap_rows // R.sq, sq=R.sq, topk=R.topk,
                                         seqlen_kv=R.seqlen_kv), device="cpu")
    O64 = O.to(torch.float64).numpy()
    dY64 = dY.to(torch.float64).numpy()
    M64 = M.to(torch.float64).numpy()
    idx_np = idx.numpy()
    pos = np.arange(c.pos0, c.pos0 + rows, dtype=np.int64)
    t0 = time.perf_counter()
    oracle.postmix_fwd(O64, M64, pos, c.nope, c.pe, c.theta)
    oracle.postmix_bwd(dY64, O64, M64, pos, c.nope, c.pe, c.theta)
    t1 = time.perf_counter()
    oracle.kv_idx_local_to_global(idx_np, R.sq, R.seqlen_kv)
    dt = time.perf_counter() - t0
    nbytes = (2 * rows * c.nh * c.d * 2 + 4 * c.nh * c.nh) + (3 * rows * c.nh * c.d * 2 + 8 * c.nh * c.nh) \
        + 2 * idx.numel() * 4
    return dt, nbytes, rows, idx.shape[0], t1 - t0


def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


def cpu_baseline(args):
    rows = int(os.environ.get("INVROPE_ORACLE_ROWS", "16384"))
    dt, nbytes, rows, idx_rows, postmix_s = oracle_sample(rows)
    return {"value": round(nbytes / dt / 1e9, 3), "unit": "GB/s", "cores": oracle_threads(),
            "kind": "oracle", "rows": rows, "postmix_s": round(postmix_s, 3),
            "sample": f"fp64 numpy oracle: fwd+bwd(dO, dM) on the first {rows} of 16384 positions "
                      f"of the production shard + remap of {idx_rows} table rows; "
                      f"{dt:.2f} s wall, scaled to algorithmic GB/s"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    rows = int(os.environ.get("INVROPE_ORACLE_ROWS", "256"))
    times = []
    nbytes = 0
    for _ in range(args.warmup):
        oracle_sample(rows)
    for _ in range(args.steps):
        dt, nbytes, rows, idx_rows, _ = oracle_sample(rows)
        times.append(dt)
    sec = statistics.mean(times)
    value = nbytes / sec / 1e9
    c = W.PROD
    line = {
        "impl": "reference",
        "metric": "fused inv-RoPE+postmix fwd/bwd us and HBM GB/s (% of roof), sq=16384 nh=64",
        "value": round(value, 3),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (same recipe as the GPU arm)",
        "config": {"workload": "production shard fwd+bwd + KV index remap, bounded sample "
                               f"({rows} of {c.sq} positions per step)",
                   "sq": c.sq, "nh": c.nh, "nope": c.nope, "pe": c.pe, "pos0": c.pos0},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "kind": "oracle",
                         "cores": oracle_threads(),
                         "sample": f"{rows} positions per step + the proportional remap slice"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=370)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
