"""Whole-layer GPU parity (forward and backward) against the C++ CPU oracle
(oracle/moe_oracle.cpp), at sizes the oracle finishes in seconds that still
span several tiles, ragged per-expert segments, partial N tiles and capacity
drops.

Both sides start from the same seeded inputs.  With learned routing the GPU
computes the router product in fp32 on the tensor cores and the oracle in
fp64 (rounded to fp32): the GPU logits are checked against the oracle's
within a tolerance, and the oracle then runs the layer on the GPU's own fp32
logits, so routing and permutation are compared bit for bit and every output
and gradient for every token and expert (tests/gpu_util.py)."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from oracle import moe_oracle_cpp as orc_cpp
from synth import workloads
from tests.gpu_util import assert_close, compare_layer, host_f64, oracle_reference, upload

pytestmark = pytest.mark.gpu


CASES = {
    # name: workload (T, d, E, k, H, Hs, routing, zipf, capacity_factor)
    "tiny": workloads.WORKLOADS["tiny"],
    "shared_ragged": workloads.custom("shared_ragged", T=700, d=256, E=16, k=4, H=256, Hs=128),
    "zipf_capacity": workloads.custom("zipf_capacity", T=700, d=256, E=16, k=2, H=256, Hs=128, zipf_bias=True,
                                      capacity_factor=1.25),
    "random_many_experts": workloads.custom("random_many_experts", T=512, d=256, E=64, k=4, H=128, Hs=128,
                                            routing="random"),
    "partial_tiles": workloads.custom("partial_tiles", T=300, d=384, E=8, k=2, H=384, Hs=384),
    # every buffer below 128 KiB: all per-expert tensor maps from the one-row class
    "micro_small_maps": workloads.custom("micro_small_maps", T=24, d=256, E=8, k=2, H=128, Hs=128),
    # the largest E and k: most experts hold 0-6 rows
    "e256_k8": workloads.custom("e256_k8", T=64, d=256, E=256, k=8, H=128, Hs=0),
    "single_token": workloads.custom("single_token", T=1, d=256, E=8, k=2, H=128, Hs=128),
    # capacity far below the load: C = 44 rows per expert, three quarters of
    # the (token, slot) pairs dropped, most experts exactly full
    "heavy_drops": workloads.custom("heavy_drops", T=700, d=256, E=16, k=4, H=256, Hs=128, capacity_factor=0.25),
    # k = E: every token in every expert (all segments T rows long)
    "k_equals_E": workloads.custom("k_equals_E", T=100, d=256, E=8, k=8, H=128, Hs=0),
}


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_routing_grouped_moe_gb300 import _binding
    return _binding


def run_layer(w, inp, poison=False):
    from top_routing_grouped_moe_gb300.layer import MoELayer
    dev = upload(inp)
    layer = MoELayer(w.T, w.d, w.E, w.k, w.H, w.Hs, w.capacity)
    if poison:
        # every floating-point buffer the path writes, and the workspace
        # (all bytes 0xFF: NaN as fp32 and bf16), starts as NaN, so a read of a
        # row that no kernel wrote (e.g. past the kept rows under a capacity
        # drop) shows up in the results.  Index buffers are left as allocated;
        # the workspace's index scratch is written before it is read.
        for v in vars(layer).values():
            if isinstance(v, torch.Tensor) and v.is_floating_point():
                v.fill_(float("nan"))
        layer.ws.fill_(0xFF)
    layer.forward(dev["x"], dev, logits_in=dev.get("logits_in"))
    layer.backward(dev["x"], dev["dY"], dev, learned_router=w.routing == "learned")
    torch.cuda.synchronize()
    return layer


@pytest.mark.parametrize("name", list(CASES))
def test_layer_forward_backward_parity(B, name):
    w = CASES[name]
    if not w.backward:
        w = workloads.custom(w.name, T=w.T, d=w.d, E=w.E, k=w.k, H=w.H, Hs=w.Hs, routing=w.routing,
                             zipf_bias=w.zipf_bias, capacity_factor=w.capacity_factor, backward=True)
    inp = workloads.make_inputs(w)
    layer = run_layer(w, inp)
    assert B.moe_device_status() == 0
    _, ref, refb, _ = oracle_reference(w, inp, layer, impl=orc_cpp)
    compare_layer(w, inp, layer, ref, refb)


@pytest.mark.parametrize("name", ["zipf_capacity", "partial_tiles", "heavy_drops"])
def test_unwritten_rows_never_leak(B, name):
    """All output and scratch buffers filled with NaN before the step: rows
    past the kept ones (capacity drop) and past each tile's valid rows are
    read by the tensor-core loads but must never reach a result."""
    w = CASES[name]
    w = workloads.custom(w.name, T=w.T, d=w.d, E=w.E, k=w.k, H=w.H, Hs=w.Hs, routing=w.routing,
                         zipf_bias=w.zipf_bias, capacity_factor=w.capacity_factor, backward=True)
    inp = workloads.make_inputs(w)
    layer = run_layer(w, inp, poison=True)
    assert B.moe_device_status() == 0
    _, ref, refb, _ = oracle_reference(w, inp, layer, impl=orc_cpp)
    compare_layer(w, inp, layer, ref, refb)


def test_layer_is_deterministic(B):
    w = workloads.custom("det", T=700, d=256, E=16, k=4, H=256, Hs=128)
    inp = workloads.make_inputs(w)
    a = run_layer(w, inp)
    ya, dxa, dwa = a.y.clone(), a.dx.clone(), a.dW_g.clone()
    b = run_layer(w, inp)
    assert torch.equal(ya.view(torch.int16), b.y.view(torch.int16))
    assert torch.equal(dxa.view(torch.int16), b.dx.view(torch.int16))
    assert torch.equal(dwa.view(torch.int16), b.dW_g.view(torch.int16))


def test_empty_experts_get_zero_weight_gradients(B):
    """All tokens routed (random routing) to 4 of 32 experts: the other 28 have
    no rows, and their dW must be exactly zero."""
    from synth import gen
    w = workloads.custom("empty", T=256, d=256, E=32, k=4, H=128, Hs=0, routing="random")
    inp = workloads.make_inputs(w)
    l = np.full((w.T, w.E), -np.inf, dtype=np.float32)
    l[:, [3, 7, 20, 31]] = gen.random_logits(w.T, 4, tensor=400)
    inp["logits_in"] = l
    layer = run_layer(w, inp)
    used = np.zeros(w.E, dtype=bool)
    used[[3, 7, 20, 31]] = True
    for name in ("dW_g", "dW_u", "dW_d"):
        v = getattr(layer, name).float().cpu().numpy()
        assert np.all(v[~used] == 0.0), name
        assert np.all(np.abs(v[used]).sum(axis=(1, 2)) > 0), name
    ref = orc.layer_forward(orc.inputs_to_f64(inp), w.k, 0)
    assert_close("y", host_f64(layer.y), ref["y"])
