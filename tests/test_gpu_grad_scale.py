"""Gradient scale: the backward's fp16 sum terms (dx_perm, dx_s and the
router's term) are stored divided by 2^e, e = floor(log2 max|dY|), and the
unpermute reduce multiplies the fp32 sum by 2^e again.  Every other step of
the backward is fp32 arithmetic or a bf16 rounding, which commute with a
power-of-two scaling, so the whole backward is exactly scale-invariant: with
dY times 2^-20 (|dY| about 1e-6, far below fp16's normal range, as a loss
averaged over many tokens gives), every gradient is the unscaled run's times
2^-20 bit for bit and the stored terms are the same bits.  Without the scale
word the terms would fall into fp16's subnormals and dx would lose most of
its precision (checked as the contrast)."""
import pytest
import torch

from synth import workloads
from tests.gpu_util import upload
from tests.test_gpu_determinism import CASES, step

pytestmark = pytest.mark.gpu

SHIFT = -20
GRADS = ["dgates", "dW_d", "dW_g", "dW_u", "dWs_d", "dWs_g", "dWs_u", "dlogits", "dW_r", "dx"]
TERMS = ["dx_perm", "dx_s"]  # stored divided by 2^e: the same bits at any scale


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_routing_grouped_moe_gb300 import _binding
    return _binding


def grads(layer, R):
    out = {}
    for n in GRADS + TERMS:
        t = getattr(layer, n, None)
        if t is None:
            continue
        out[n] = (t[:R] if n == "dx_perm" else t).clone()
    return out


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("fused", [False, True], ids=["unfused", "fused"])
def test_backward_is_exact_under_power_of_two_gradient_scaling(B, name, fused):
    from top_routing_grouped_moe_gb300.layer import MoELayer
    w = CASES[name]
    dev = upload(workloads.make_inputs(w))
    layer = MoELayer(w.T, w.d, w.E, w.k, w.H, w.Hs, w.capacity, fused=fused)
    step(layer, w, dev)
    torch.cuda.synchronize()
    R = int(layer.offsets[-1].item())
    ref = grads(layer, R)
    small = dict(dev)
    small["dY"] = (dev["dY"].float() * 2.0 ** SHIFT).to(torch.bfloat16)  # exact: a power of two
    step(layer, w, small)
    torch.cuda.synchronize()
    assert B.moe_device_status() == 0
    got = grads(layer, R)
    for n in GRADS:
        if n in ref:
            want = ref[n].double() * 2.0 ** SHIFT
            assert torch.equal(got[n].double(), want), f"{n}: not the unscaled gradient times 2^{SHIFT}"
    for n in TERMS:
        if n in ref:
            assert torch.equal(got[n].view(torch.int16), ref[n].view(torch.int16)), f"{n}: stored terms differ"

    # contrast: the same small gradient with unscaled fp16 terms
    if fused:
        return
    layer.dx_scale, keep = None, layer.dx_scale
    try:
        step(layer, w, small)
        torch.cuda.synchronize()
    finally:
        layer.dx_scale = keep
    exact = ref["dx"].double() * 2.0 ** SHIFT
    rel = (layer.dx.double() - exact).norm() / exact.norm()
    assert rel > 1e-2, f"unscaled fp16 terms at |dY| ~ 1e-6 unexpectedly accurate (rel {rel:.2e})"
