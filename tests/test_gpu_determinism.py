"""Determinism and graph capture of the whole layer step.

Every output element is owned by one tile with a fixed summation order, and
the dynamic tile schedule of the weight gradients only changes which CTA
computes a tile, so two runs of the same step give bit-identical results.
The step allocates nothing and never waits on the host, so it can be
captured in a CUDA graph (the bench times it that way); a replay gives the
same bits as the eager calls."""
import pytest
import torch

from synth import workloads
from tests.gpu_util import upload

pytestmark = pytest.mark.gpu

OUTPUTS = ["logits", "idx", "gates", "counts", "offsets", "row_of_slot", "y", "h", "au", "o_perm", "dgates",
           "dx_perm", "dW_g", "dW_u", "dW_d", "dWs_g", "dWs_u", "dWs_d", "dlogits", "dW_r", "dx"]
CASES = {
    "learned_shared": workloads.custom("learned_shared", T=700, d=256, E=16, k=4, H=256, Hs=128, backward=True),
    "zipf_capacity": workloads.custom("zipf_capacity", T=700, d=256, E=16, k=2, H=256, Hs=128, zipf_bias=True,
                                      capacity_factor=1.25, backward=True),
}


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_routing_grouped_moe_gb300 import _binding
    return _binding


ROW_SPACE = ("h", "au", "o_perm", "dx_perm")  # [T*k, ...]: only rows [0, R) are written


def snapshot(layer):
    """The written part of every output (a fused layer's o_perm holds the
    expert outputs by slot, dropped slots unwritten: y covers it)."""
    R = int(layer.offsets[-1].item())
    out = {}
    for n in OUTPUTS:
        t = getattr(layer, n, None)
        if t is None or (n == "o_perm" and layer.fused):
            continue
        out[n] = (t[:R] if n in ROW_SPACE else t).clone()
    return out


def clear(layer):
    R = int(layer.offsets[-1].item())
    for n in OUTPUTS:
        t = getattr(layer, n, None)
        if t is not None:
            (t[:R] if n in ROW_SPACE else t).zero_()


def step(layer, w, dev, stream=None):
    layer.forward(dev["x"], dev, logits_in=dev.get("logits_in"), stream=stream)
    layer.backward(dev["x"], dev["dY"], dev, learned_router=w.routing == "learned", stream=stream)


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("fused", [False, True])
def test_step_is_bit_reproducible_and_graph_capturable(B, name, fused):
    from top_routing_grouped_moe_gb300.layer import MoELayer
    w = CASES[name]
    dev = upload(workloads.make_inputs(w))
    layer = MoELayer(w.T, w.d, w.E, w.k, w.H, w.Hs, w.capacity, fused=fused)
    step(layer, w, dev)
    torch.cuda.synchronize()
    first = snapshot(layer)
    step(layer, w, dev)
    torch.cuda.synchronize()
    second = snapshot(layer)
    assert B.moe_device_status() == 0
    for n in first:
        assert torch.equal(first[n].view(torch.uint8), second[n].view(torch.uint8)), f"{n}: run to run"
    # the same step captured once and replayed, after the outputs are cleared
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(layer, w, dev, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    clear(layer)
    g.replay()
    torch.cuda.synchronize()
    assert B.moe_device_status() == 0
    replay = snapshot(layer)
    for n in first:
        assert torch.equal(first[n].view(torch.uint8), replay[n].view(torch.uint8)), f"{n}: graph replay"
