"""The fused path (moe_grouped_swiglu_fused, the gather mode of
moe_grouped_swiglu_bwd): the permutation fused into the GEMMs' operand loads
(TMA row gathers from x and dY) and the combine fused into the shared
expert's down-projection epilogue.

Each case runs the fused layer against the C++ oracle (every output and
gradient, routing bit-exact) and against the unfused layer on the same
inputs.  Both read the same operand values in the same order, so the
forward outputs and the GEMM gradients are identical (value equality; y by
construction, since the fused epilogue repeats the combine's operations in
its order).  The gate gradient is the one exception: the gathering GEMMs run
on single CTAs, whose tiles sum each row's gate-gradient partial over 256
columns where the CTA pairs' half tiles sum two halves of 128, so dgates --
and dlogits, dW_r and dx, which take it in -- differ by fp32 rounding."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle_cpp as orc_cpp
from synth import workloads
from tests.gpu_util import compare_layer, oracle_reference, upload

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": workloads.WORKLOADS["tiny"],
    "shared_ragged": workloads.custom("shared_ragged", T=700, d=256, E=16, k=4, H=256, Hs=128),
    "zipf_capacity": workloads.custom("zipf_capacity", T=700, d=256, E=16, k=2, H=256, Hs=128, zipf_bias=True,
                                      capacity_factor=1.25),
    "random_many_experts": workloads.custom("random_many_experts", T=512, d=256, E=64, k=4, H=128, Hs=128,
                                            routing="random"),
    "partial_tiles": workloads.custom("partial_tiles", T=300, d=384, E=8, k=2, H=384, Hs=384),
    "micro_small_maps": workloads.custom("micro_small_maps", T=24, d=256, E=8, k=2, H=128, Hs=128),
    # no shared expert: the combine runs as its own pass over the slot-ordered outputs
    "e256_k8_no_shared": workloads.custom("e256_k8", T=64, d=256, E=256, k=8, H=128, Hs=0),
    "single_token": workloads.custom("single_token", T=1, d=256, E=8, k=2, H=128, Hs=128),
    # several 256-row tiles per expert, a ragged last tile (M = 128 pair tiles)
    "long_groups": workloads.custom("long_groups", T=1500, d=512, E=8, k=2, H=256, Hs=256),
}


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_routing_grouped_moe_gb300 import _binding
    return _binding


def with_backward(w):
    if w.backward:
        return w
    return workloads.custom(w.name, T=w.T, d=w.d, E=w.E, k=w.k, H=w.H, Hs=w.Hs, routing=w.routing,
                            zipf_bias=w.zipf_bias, capacity_factor=w.capacity_factor, backward=True)


def run(w, dev, fused, recompute=False, poison=False):
    from top_routing_grouped_moe_gb300.layer import MoELayer
    layer = MoELayer(w.T, w.d, w.E, w.k, w.H, w.Hs, w.capacity, fused=fused, recompute=recompute)
    if poison:
        # every floating-point buffer and the workspace start as NaN: a read
        # of anything no kernel wrote (a dropped slot's output row, a row past
        # a group's end) shows up in the results
        for v in vars(layer).values():
            if isinstance(v, torch.Tensor) and v.is_floating_point():
                v.fill_(float("nan"))
        layer.ws.fill_(0xFF)
    layer.forward(dev["x"], dev, logits_in=dev.get("logits_in"))
    layer.backward(dev["x"], dev["dY"], dev, learned_router=w.routing == "learned")
    torch.cuda.synchronize()
    return layer


OUTPUTS = ["y", "h", "au", "au_s", "h_s", "gates", "dx_perm", "dx_s", "dW_g", "dW_u", "dW_d", "dWs_g", "dWs_u",
           "dWs_d"]
# (name, rtol, atol as a fraction of the tensor's largest magnitude): the
# fp32 rounding of the gate gradient's partial sums (sums of H products,
# near zero where they cancel); dx additionally its bf16 rounding
NEAR = [("dgates", 1e-4, 1e-5), ("dlogits", 1e-4, 1e-5), ("dW_r", 1e-4, 1e-5), ("dx", 1e-2, 1e-3)]


def near_close(n, a, b, rtol, atol_frac):
    a, b = a.float(), b.float()
    scale = float(b.abs().max())
    diff = float((a - b).abs().max())
    torch.testing.assert_close(a, b, rtol=rtol, atol=atol_frac * scale + 1e-7,
                               msg=f"{n}: max |fused - unfused| {diff:.3e}, max |unfused| {scale:.3e}")


def assert_near(w, a, b):
    for n, rtol, atol in NEAR:
        if n == "dW_r" and w.routing != "learned":
            continue
        near_close(n, getattr(a, n), getattr(b, n), rtol, atol)


def assert_same(w, a, b, names):
    R = int(a.offsets[-1].item())
    for n in names:
        ta, tb = getattr(a, n, None), getattr(b, n, None)
        if ta is None or tb is None:
            assert ta is None and tb is None, n
            continue
        if n in ("h", "au", "dx_perm"):
            ta, tb = ta[:R], tb[:R]
        if n == "dW_r" and w.routing != "learned":
            continue
        assert torch.equal(ta, tb), f"{n}: fused differs from unfused"


@pytest.mark.parametrize("name", list(CASES))
def test_fused_layer_parity(B, name):
    w = with_backward(CASES[name])
    inp = workloads.make_inputs(w)
    dev = upload(inp)
    fused = run(w, dev, fused=True, poison=True)
    assert B.moe_device_status() == 0
    assert fused.x_perm is None and fused.dY_perm is None and fused.s is None
    _, ref, refb, _ = oracle_reference(w, inp, fused, impl=orc_cpp)
    compare_layer(w, inp, fused, ref, refb)

    plain = run(w, dev, fused=False)
    assert B.moe_device_status() == 0
    assert_same(w, fused, plain, OUTPUTS)
    assert_near(w, fused, plain)
    # expert outputs: by slot in the fused layer, by permuted row in the other
    R = int(plain.offsets[-1].item())
    slots = plain.slot_of_row[:R].long()
    assert torch.equal(fused.o_perm[slots], plain.o_perm[:R])


@pytest.mark.parametrize("name", ["shared_ragged", "zipf_capacity", "e256_k8_no_shared"])
def test_fused_recompute(B, name):
    """Fused forward without saved a | u, rebuilt by the fused recompute:
    the same gradients as the fused layer that saved them."""
    w = with_backward(CASES[name])
    dev = upload(workloads.make_inputs(w))
    saved = run(w, dev, fused=True)
    rec = run(w, dev, fused=True, recompute=True)
    assert B.moe_device_status() == 0
    assert_same(w, rec, saved, OUTPUTS + [n for n, _, _ in NEAR])


def test_fused_entry_point_checks(B):
    """Argument checks of the fused calls (no kernel runs)."""
    w = CASES["tiny"]
    T, d, E, k, H, Hs = w.T, w.d, w.E, w.k, w.H, w.Hs
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.MoEError) as e:
        B.moe_grouped_swiglu_fused(None, z, z, z, z, T, d, E, k, H, Hs, z, z, z, z, z, z, None, z, z, None, z, z)
    assert e.value.status == B.MOE_ERR_INVALID_ARG
    # x_perm given without dY_perm (or the reverse) is neither mode
    with pytest.raises(B.MoEError) as e:
        B.moe_grouped_swiglu_bwd(None, z, z, z, z, z, z, z, z, z, T, d, E, k, H, Hs, z, z, z, z, z, z, z, z, z, z,
                                 z, z, z, z, z, z, 1 << 30)
    assert e.value.status == B.MOE_ERR_INVALID_ARG
