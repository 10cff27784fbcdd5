"""Activation recompute for the backward: moe_grouped_swiglu_recompute must
rebuild exactly (bit for bit) the fp32 a | u that the forward would have
saved, and a layer run with recompute must give a backward identical to one
that saved them, and so match the oracle."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from synth import workloads
from tests.gpu_util import compare_layer, oracle_reference, upload

pytestmark = pytest.mark.gpu

CASES = {
    "shared_ragged": workloads.custom("shared_ragged", T=700, d=256, E=16, k=4, H=256, Hs=128),
    "zipf_capacity": workloads.custom("zipf_capacity", T=700, d=256, E=16, k=2, H=256, Hs=128, zipf_bias=True,
                                      capacity_factor=1.25),
    "no_shared_partial": workloads.custom("no_shared_partial", T=300, d=384, E=8, k=2, H=384, Hs=0),
}


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_routing_grouped_moe_gb300 import _binding
    return _binding


def run(w, dev, recompute):
    from top_routing_grouped_moe_gb300.layer import MoELayer
    layer = MoELayer(w.T, w.d, w.E, w.k, w.H, w.Hs, w.capacity, recompute=recompute)
    if recompute:
        # nothing the forward might have left behind: a|u start as NaN
        layer.au.fill_(float("nan"))
        if layer.au_s is not None:
            layer.au_s.fill_(float("nan"))
    layer.forward(dev["x"], dev, logits_in=dev.get("logits_in"))
    torch.cuda.synchronize()
    au_after_fwd = layer.au.clone()
    layer.backward(dev["x"], dev["dY"], dev, learned_router=w.routing == "learned")
    torch.cuda.synchronize()
    return layer, au_after_fwd


def bits(t):
    return t.contiguous().view(torch.int32).cpu().numpy()


@pytest.mark.parametrize("name", list(CASES))
def test_recompute_is_bit_identical_to_the_saved_activations(B, name):
    w = CASES[name]
    dev = upload(workloads.make_inputs(w))
    saved, _ = run(w, dev, recompute=False)
    R = int(saved.offsets[-1])
    au = torch.full_like(saved.au, float("nan"))
    au_s = torch.full_like(saved.au_s, float("nan")) if w.Hs else None
    B.moe_grouped_swiglu_recompute(saved.x_perm, saved.offsets, dev["x"], w.T, w.d, w.E, w.k, w.H, w.Hs,
                                   dev["W_g"], dev["W_u"], dev.get("Ws_g"), dev.get("Ws_u"), au, au_s)
    torch.cuda.synchronize()
    assert B.moe_device_status() == 0
    assert np.array_equal(bits(au[:R]), bits(saved.au[:R]))
    if w.Hs:
        assert np.array_equal(bits(au_s), bits(saved.au_s))
    # rows past the kept ones are not written
    assert torch.isnan(au[R:]).all()


@pytest.mark.parametrize("name", list(CASES))
def test_layer_with_recompute(B, name):
    w = CASES[name]
    inp = workloads.make_inputs(w)
    dev = upload(inp)
    saved, _ = run(w, dev, recompute=False)
    rec, au_after_fwd = run(w, dev, recompute=True)
    assert B.moe_device_status() == 0
    R = int(rec.offsets[-1])
    # the forward of the recompute layer saved nothing
    assert torch.isnan(au_after_fwd[:R]).all()
    # identical forward and backward results
    for n in ("y", "dx", "dW_g", "dW_u", "dW_d", "dWs_g", "dWs_u", "dWs_d", "dgates", "dlogits", "dW_r"):
        a, b = getattr(saved, n), getattr(rec, n)
        if a is None:
            continue
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b), n
    _, ref, refb, _ = oracle_reference(w, inp, rec)
    compare_layer(w, inp, rec, ref, refb)
