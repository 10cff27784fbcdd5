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


# Twice bf16's unit roundoff: the bound on one bf16 rounding (round to nearest
# even, relative error at most 2^-9) with room for the fp32 accumulation.
BF16_ROUNDING = 2.0 ** -8


def bf16_operand_allowance(w, f64, ref, refb):
    """Per-element bounds on what the GEMM operands the design rounds to bf16
    (h into the down projection, the routed rows' da|du into the gate/up
    dgrad) can move each output: |sum_j (A~_j - A_j) B_j| <= 2^-8 sum_j |A_j| |B_j|,
    with A the oracle's float64 operand, propagated through the combine and
    the unpermute sums.  The shared expert's da|du is split (hi + lo) and
    adds nothing."""
    T, k, E = w.T, w.k, w.E
    off = ref["offsets"]
    R = int(off[-1])
    o_a = np.zeros((R, w.d))
    dxp_a = np.zeros((R, w.d))
    for e in range(E):
        r0, r1 = int(off[e]), int(off[e + 1])
        if r1 == r0:
            continue
        Wg, Wu, Wd = f64["W_g"][e], f64["W_u"][e], f64["W_d"][e]  # [H,d], [H,d], [d,H]
        o_a[r0:r1] = BF16_ROUNDING * (np.abs(ref["h"][r0:r1]) @ np.abs(Wd).T)
        a, u = ref["a"][r0:r1], ref["u"][r0:r1]
        dh = refb["dO"][r0:r1] @ Wd  # the gate-weighted upstream gradient through W_d
        sg = 1.0 / (1.0 + np.exp(-a))
        da = dh * u * sg * (1.0 + a * (1.0 - sg))
        du = dh * a * sg
        dxp_a[r0:r1] = BF16_ROUNDING * (np.abs(da) @ np.abs(Wg) + np.abs(du) @ np.abs(Wu))
    s_a = BF16_ROUNDING * (np.abs(ref["h_s"]) @ np.abs(f64["Ws_d"]).T) if w.Hs else np.zeros((T, w.d))
    rows = ref["row_of_slot"].reshape(T, k)
    gates = np.asarray(ref["gates"], dtype=np.float64).reshape(T, k)
    y_a = s_a.copy()
    dx_a = np.zeros((T, w.d))
    for slot in range(k):
        kept = rows[:, slot] >= 0
        y_a[kept] += np.abs(gates[kept, slot])[:, None] * o_a[rows[kept, slot]]
        dx_a[kept] += dxp_a[rows[kept, slot]]
    return {"o_perm": o_a, "s": s_a, "y": y_a, "dx_perm": dxp_a, "dx": dx_a}


def test_wide_layer_within_the_bf16_operand_rounding(B):
    """d = 8192, H = 2048, wider than any layer configuration (128 K steps per
    gate/up tile, 32 column tiles of the down projection).  Its outputs grow
    with d (RMS about 2), and the bf16 rounding of h and of the routed da|du,
    relative 2^-9, then exceeds the bar's absolute 1e-2 on a few hundred of
    millions of elements (relative Frobenius stays 1.7e-3).  Every output and
    gradient must still be within the bar plus that rounding's own bound, and
    routing and permutation bit-exact."""
    w = workloads.custom("wide", T=256, d=8192, E=8, k=2, H=2048, Hs=1024)
    inp = workloads.make_inputs(w)
    layer = run_layer(w, inp)
    assert B.moe_device_status() == 0
    f64, ref, refb, _ = oracle_reference(w, inp, layer, impl=orc_cpp)
    compare_layer(w, inp, layer, ref, refb, allow=bf16_operand_allowance(w, f64, ref, refb))
