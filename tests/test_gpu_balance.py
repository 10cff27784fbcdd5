"""GPU parity of the router balance loss (auxiliary load-balancing loss)
against the CPU oracle: the kernel on its own over expert counts that take
every softmax width (E = 8 ... 256, ragged token counts, -inf logits of
random routing), and inside the layer, where its gradient must reach
dlogits, dW_r and dx."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from synth import gen, workloads
from tests.gpu_util import compare_layer, oracle_reference, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from top_routing_grouped_moe_gb300 import _binding
    return _binding


def _logits(T, E, k, kind, seed):
    if kind == "random_routing":
        return gen.random_routing_logits(T, E, k, base=gen.BASE_SEED + seed).astype(np.float32)
    rng = np.random.default_rng(seed)
    return (rng.normal(size=(T, E)) * 2.0).astype(np.float32)


def _run(B, l32, idx, E, k, alpha):
    T = l32.shape[0]
    counts = np.bincount(idx.ravel().astype(np.int64), minlength=E).astype(np.int32)
    ws_bytes = B.moe_workspace_size(T, 64, E, k, 128, 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    P = torch.empty(E, dtype=torch.float32, device="cuda")
    dl = torch.empty(T, E, dtype=torch.float32, device="cuda")
    B.moe_router_balance_loss(torch.from_numpy(l32).cuda(), torch.from_numpy(counts).cuda(), T, E, k, alpha, loss,
                              P, dl, ws, ws_bytes)
    torch.cuda.synchronize()
    return float(loss.item()), P.cpu().numpy().astype(np.float64), dl.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("T,E,k,kind", [(1000, 64, 4, "normal"), (77, 8, 2, "normal"), (300, 256, 8, "normal"),
                                        (129, 40, 3, "normal"), (1000, 64, 4, "random_routing")])
def test_balance_loss_kernel_parity(B, T, E, k, kind):
    l32 = _logits(T, E, k, kind, seed=T + E)
    idx, _ = orc.route_topk(l32, k)
    alpha = 0.05
    L, f, P, dl = orc.balance_loss(l32.astype(np.float64), idx, E, alpha)
    gL, gP, gdl = _run(B, l32, idx, E, k, alpha)
    assert B.moe_device_status() == 0
    assert abs(gL - L) <= 1e-6 * abs(L) + 1e-9, (gL, L)
    np.testing.assert_allclose(gP, P, rtol=1e-5, atol=1e-7)
    # f_j - sum_e f_e p_e cancels for some entries: fp32 leaves ~1e-7 of the largest entry there
    np.testing.assert_allclose(gdl, dl, rtol=1e-4, atol=1e-6 * np.abs(dl).max())
    # deterministic (fixed-order reductions)
    gL2, gP2, gdl2 = _run(B, l32, idx, E, k, alpha)
    assert gL2 == gL and np.array_equal(gP2, gP) and np.array_equal(gdl2, gdl)


@pytest.mark.parametrize("routing", ["learned", "random"])
def test_balance_loss_in_the_layer(B, routing):
    """The layer with the loss on: its value, and its gradient inside dlogits,
    dW_r (learned routing) and dx, against the oracle with the same term
    added; the difference of two GPU runs (alpha on / off) isolates the
    added term in dlogits and dW_r exactly."""
    from top_routing_grouped_moe_gb300.layer import MoELayer
    w = workloads.custom("lbl_" + routing, T=700, d=256, E=16, k=4, H=256, Hs=128, routing=routing)
    inp = workloads.make_inputs(w)
    alpha = 10.0  # large, so that the isolated term stands well above fp32 rounding of the rest
    dev = upload(inp)
    layers = {}
    for a in (0.0, alpha):
        L_ = MoELayer(w.T, w.d, w.E, w.k, w.H, w.Hs, w.capacity, balance_alpha=a)
        L_.forward(dev["x"], dev, logits_in=dev.get("logits_in"))
        L_.backward(dev["x"], dev["dY"], dev, learned_router=routing == "learned")
        layers[a] = L_
    torch.cuda.synchronize()
    assert B.moe_device_status() == 0
    layer = layers[alpha]

    f64, ref, refb, _ = oracle_reference(w, inp, layer)
    Lr, fr, Pr, dlr = orc.balance_loss(ref["logits"], ref["idx"], w.E, alpha)
    assert abs(float(layer.lbl_loss.item()) - Lr) <= 1e-4 * abs(Lr)
    np.testing.assert_allclose(layer.lbl_P.cpu().numpy(), Pr, rtol=1e-4, atol=1e-6)

    # the added term, isolated: the difference of two fp32 sums carries a few
    # ulps of the unchanged term
    dl0 = layers[0.0].dlogits.cpu().numpy().astype(np.float64)
    ddl = layer.dlogits.cpu().numpy().astype(np.float64) - dl0
    np.testing.assert_allclose(ddl, dlr, rtol=2e-3, atol=4 * 2.0 ** -24 * np.abs(dl0).max())
    if routing == "learned":
        ddw = (layer.dW_r - layers[0.0].dW_r).cpu().numpy().astype(np.float64)
        ref_dw = dlr.T @ f64["x"]
        err = np.linalg.norm(ddw - ref_dw) / np.linalg.norm(ref_dw)
        assert err < 5e-3, err

    # the whole backward with the term included, at the layer tolerance
    refb["dlogits"] = refb["dlogits"] + dlr
    if routing == "learned":
        refb["dW_r"] = refb["dW_r"] + dlr.T @ f64["x"]
        refb["dx"] = refb["dx"] + dlr @ f64["W_r"]
    compare_layer(w, inp, layer, ref, refb)
