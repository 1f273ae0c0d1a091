"""The library's calls on several streams at once, and inside a captured CUDA
graph: both must give the same bits as plain calls on one stream. The forward
and the remap claim work from a per-launch counter slot and the backward's
reduction is a programmatic dependent launch, so these are the paths that
concurrency and capture could disturb. A launch that finds its slot held by
another launch must report it rather than share the counter. Needs a GB300
(sm_103a)."""

import pytest
import torch

import partial_inverse_rope_gb300 as ir
from gpu_helpers import ensure_built, make_inputs
from partial_inverse_rope_gb300 import binding

pytestmark = pytest.mark.gpu

SHAPE = (2048, 16, 448, 64)  # sq, nh, nope, pe (the mid config's shape)


@pytest.fixture(scope="module", autouse=True)
def built():
    ensure_built()
    yield
    assert ir.invrope_take_device_fault() == 0, "a kernel wait ran out during the tests"


def _case(seed):
    sq, nh, nope, pe = SHAPE
    O, dY, M = make_inputs(sq, nh, nope, pe, seed=seed)
    g = torch.Generator(device="cuda").manual_seed(seed)
    idx = torch.randint(-1, 4096, (4 * 512, 256), generator=g, device="cuda", dtype=torch.int32)
    return O, dY, M, idx


def _outputs(O, idx):
    nh = O.shape[1]
    ws = torch.empty(ir.invrope_postmix_bwd_workspace_bytes(*SHAPE), dtype=torch.uint8, device="cuda")
    return dict(Y=torch.empty_like(O), dO=torch.empty_like(O),
                dM=torch.empty(nh, nh, dtype=torch.float32, device="cuda"),
                out=torch.empty_like(idx), ws=ws)


def _run(case, o, stream=None):
    O, dY, M, idx = case
    _, _, nope, pe = SHAPE
    ir.invrope_postmix_fwd(O, M, 7, nope, pe, Y=o["Y"], stream=stream)
    ir.invrope_postmix_bwd(dY, O, M, 7, nope, pe, dO=o["dO"], dM=o["dM"], workspace=o["ws"], stream=stream)
    ir.kv_idx_local_to_global(idx, 512, 4096, out=o["out"], stream=stream)


def _same(a, b):
    for k in ("Y", "dO", "dM", "out"):
        assert torch.equal(a[k], b[k]), k


def test_concurrent_streams_match_one_stream():
    cases = [_case(s) for s in (21, 22, 23)]
    ref = []
    for c in cases:
        o = _outputs(c[0], c[3])
        _run(c, o)
        ref.append(o)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in cases]
    outs = [_outputs(c[0], c[3]) for c in cases]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        for c, o, s in zip(cases, outs, streams):
            _run(c, o, stream=s)
    torch.cuda.synchronize()
    for r, o in zip(ref, outs):
        _same(r, o)


def test_graph_replay_matches_eager():
    case = _case(31)
    eager = _outputs(case[0], case[3])
    _run(case, eager)  # also loads the module and sets kernel attributes before capture
    torch.cuda.synchronize()
    o = _outputs(case[0], case[3])
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            _run(case, o)
    torch.cuda.synchronize()
    for _ in range(3):
        for v in o.values():
            v.zero_()
        graph.replay()
        torch.cuda.synchronize()
        _same(eager, o)


def test_graph_replay_beside_many_eager_launches():
    """A captured forward and remap keep their (capture) counter slots on every
    replay; eager launches on another stream cycle through the eager slots at
    the same time, more than 256 of them, and never meet the replay's slot."""
    case = _case(41)
    O, dY, M, idx = case
    _, _, nope, pe = SHAPE
    eager = _outputs(O, idx)
    _run(case, eager)
    torch.cuda.synchronize()
    o = _outputs(O, idx)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            ir.invrope_postmix_fwd(O, M, 7, nope, pe, Y=o["Y"])
            ir.kv_idx_local_to_global(idx, 512, 4096, out=o["out"])
    torch.cuda.synchronize()
    other = torch.cuda.Stream()
    Ys = [torch.empty_like(O) for _ in range(2)]
    outs = [torch.empty_like(idx) for _ in range(2)]
    for _ in range(3):
        o["Y"].zero_()
        o["out"].zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            graph.replay()
        with torch.cuda.stream(other):
            for k in range(300):
                ir.invrope_postmix_fwd(O, M, 7, nope, pe, Y=Ys[k % 2], stream=other)
                ir.kv_idx_local_to_global(idx, 512, 4096, out=outs[k % 2], stream=other)
        torch.cuda.synchronize()
        assert torch.equal(o["Y"], eager["Y"])
        assert torch.equal(o["out"], eager["out"])
        assert torch.equal(Ys[1], eager["Y"]) and torch.equal(outs[1], eager["out"])
    assert ir.invrope_take_device_fault() == 0


@pytest.mark.parametrize("which", ["fwd", "bwd", "remap"])
def test_busy_slot_is_reported_not_shared(which):
    """The next launch's counter slot is marked as held by a launch tag that no
    launch has (a host-side write through the test hook): that launch must
    claim nothing from it and record the busy-slot code. Taking the fault frees
    every slot, and the next call gives the bits of a plain call again. The
    backward takes a slot (from the forward's slots) when it hands out tail
    blocks, as at 4096 positions of 64 heads; the forward and the remap when
    they have more work than their first tile or chunk per thread block."""
    case = _case(43)
    O, dY, M, _ = case
    _, _, nope, pe = SHAPE
    Ob, dYb, Mb = make_inputs(4096, 64, 448, 64, seed=44)
    # a remap takes a slot only when it has more chunks than thread blocks:
    # 2048 rows x 8192 entries (4M 16-byte vectors, 2048 chunks of 2048)
    g = torch.Generator(device="cuda").manual_seed(45)
    idx = torch.randint(-1, 4096, (4 * 512, 8192), generator=g, device="cuda", dtype=torch.int32)

    def call():
        if which == "fwd":
            return ir.invrope_postmix_fwd(O, M, 7, nope, pe)
        if which == "bwd":
            return torch.cat([t.flatten().view(torch.int8) for t in
                              ir.invrope_postmix_bwd(dYb, Ob, Mb, 16384, 448, 64)])
        return ir.kv_idx_local_to_global(idx, 512, 4096)

    ref = call()
    assert ir.invrope_take_device_fault() == 0
    ir.invrope_debug_occupy_next_slot("remap" if which == "remap" else "fwd", (1 << 63) + 12345)
    call()  # finds its slot busy: output undefined
    want = {"fwd": binding.INVROPE_FAULT_SCHED_BUSY_FWD, "bwd": binding.INVROPE_FAULT_SCHED_BUSY_BWD,
            "remap": binding.INVROPE_FAULT_SCHED_BUSY_REMAP}[which]
    assert ir.invrope_take_device_fault() == want
    for _ in range(3):
        assert torch.equal(call(), ref)
    assert ir.invrope_take_device_fault() == 0


@pytest.mark.parametrize("which", ["fwd", "remap"])
def test_small_launches_take_no_slot(which):
    """A forward with at most two tiles per thread block (the tiny shape) and a
    remap with no more chunks than thread blocks claim nothing and take no
    work-counter slot: with the next slot marked busy they still run
    correctly and record no fault, and the next slot-taking launch is the
    one that finds it busy."""
    O, dY, M = make_inputs(128, 4, 48, 16, seed=46)
    small_idx = torch.randint(-1, 4096, (4 * 64, 64), device="cuda", dtype=torch.int32,
                              generator=torch.Generator(device="cuda").manual_seed(46))
    big = _case(47)
    big_idx = torch.randint(-1, 4096, (4 * 512, 8192), device="cuda", dtype=torch.int32,
                            generator=torch.Generator(device="cuda").manual_seed(47))
    _, _, nope, pe = SHAPE

    def small():
        if which == "fwd":
            return ir.invrope_postmix_fwd(O, M, 3, 48, 16)
        return ir.kv_idx_local_to_global(small_idx, 64, 4096)

    def large():
        if which == "fwd":
            return ir.invrope_postmix_fwd(big[0], big[2], 7, nope, pe)
        return ir.kv_idx_local_to_global(big_idx, 512, 4096)

    ref = small()
    assert ir.invrope_take_device_fault() == 0
    ir.invrope_debug_occupy_next_slot(which, (1 << 63) + 4321)
    for _ in range(3):
        assert torch.equal(small(), ref)
    assert ir.invrope_take_device_fault() == 0  # the slot is still marked: nothing took it
    large()  # takes the marked slot: finds it busy
    want = binding.INVROPE_FAULT_SCHED_BUSY_FWD if which == "fwd" else binding.INVROPE_FAULT_SCHED_BUSY_REMAP
    assert ir.invrope_take_device_fault() == want
