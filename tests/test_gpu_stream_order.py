"""Stream order with the caller's own work on the same stream.

Every kernel of the library is launched with programmatic stream
serialization and waits (griddepcontrol.wait) for the kernel before it to
complete before any global access, and no kernel signals its dependents
early.  So the caller's kernels around the calls stay ordered with them: a
caller kernel that writes an input just before a call is seen by it, and one
that overwrites the inputs and weights just after the last call, with no host
synchronisation in between, does not disturb the results."""
import pytest
import torch

from synth import workloads
from tests.gpu_util import upload
from tests.test_gpu_determinism import CASES, clear, snapshot, step

pytestmark = pytest.mark.gpu

WEIGHTS = ("W_r", "W_g", "W_u", "W_d", "Ws_g", "Ws_u", "Ws_d")


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_routing_grouped_moe_gb300 import _binding
    return _binding


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("fused", [False, True])
def test_caller_kernels_around_the_calls_stay_ordered(B, name, fused):
    from top_routing_grouped_moe_gb300.layer import MoELayer
    w = CASES[name]
    dev = upload(workloads.make_inputs(w))
    layer = MoELayer(w.T, w.d, w.E, w.k, w.H, w.Hs, w.capacity, fused=fused)
    step(layer, w, dev)
    torch.cuda.synchronize()
    ref = snapshot(layer)
    clear(layer)

    # private copies of the inputs and weights, filled with NaN; the caller's
    # copy kernels write the real values just before the calls that read
    # them, and NaN again just after the last call
    mine = {key: torch.full_like(v, float("nan")) for key, v in dev.items()}
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for key in mine:
            if key != "dY":
                mine[key].copy_(dev[key])
        layer.forward(mine["x"], mine, logits_in=mine.get("logits_in"), stream=s)
        mine["dY"].copy_(dev["dY"])
        layer.backward(mine["x"], mine["dY"], mine, learned_router=w.routing == "learned", stream=s)
        for key in ("x", "dY") + WEIGHTS:
            if key in mine:
                mine[key].fill_(float("nan"))
    torch.cuda.synchronize()
    assert B.moe_device_status() == 0
    got = snapshot(layer)
    for n in ref:
        assert torch.equal(ref[n].view(torch.uint8), got[n].view(torch.uint8)), n


def test_launch_timing_eager_and_inside_a_graph(B):
    """The library's timing marks: eager calls and a captured graph of the
    same step see the same launches in the same order, and the graph's marks
    are recorded again at each replay (times that add up to more than 0)."""
    from top_routing_grouped_moe_gb300.layer import MoELayer
    w = CASES["learned_shared"]
    dev = upload(workloads.make_inputs(w))
    layer = MoELayer(w.T, w.d, w.E, w.k, w.H, w.Hs, w.capacity)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with B.LaunchTimer(capacity=64, stream=s) as tm:
        step(layer, w, dev, stream=s)
    torch.cuda.synchronize()
    eager = tm.launches()
    assert len(eager) >= 10 and all(ms >= 0 for _, ms in eager) and sum(ms for _, ms in eager) > 0
    tg = B.LaunchTimer(capacity=64, stream=s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        with tg:
            step(layer, w, dev, stream=s)
    torch.cuda.synchronize()
    names = [n for n, _ in eager if not n.startswith("memset")]
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        got = tg.launches()
        assert [n for n, _ in got if not n.startswith("memset")] == names
        assert all(ms >= 0 for _, ms in got) and sum(ms for _, ms in got) > 0
    assert B.moe_device_status() == 0


def test_two_layers_on_two_streams_at_once(B):
    """Two layers (their own buffers and workspaces) stepping on two streams
    at the same time -- persistent GEMMs and programmatic launches of both
    interleaving on the SMs -- give the same bits as when each steps alone."""
    from top_routing_grouped_moe_gb300.layer import MoELayer
    from tests.test_gpu_determinism import snapshot
    ws = [CASES["learned_shared"], CASES["zipf_capacity"]]
    devs = [upload(workloads.make_inputs(w)) for w in ws]
    layers = [MoELayer(w.T, w.d, w.E, w.k, w.H, w.Hs, w.capacity) for w in ws]
    alone = []
    for w, dev, layer in zip(ws, devs, layers):
        step(layer, w, dev)
        torch.cuda.synchronize()
        alone.append(snapshot(layer))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        for w, dev, layer, s in zip(ws, devs, layers, streams):
            with torch.cuda.stream(s):
                step(layer, w, dev, stream=s)
    torch.cuda.synchronize()
    assert B.moe_device_status() == 0
    for layer, ref in zip(layers, alone):
        got = snapshot(layer)
        for n in ref:
            assert torch.equal(got[n].view(torch.uint8), ref[n].view(torch.uint8)), n
