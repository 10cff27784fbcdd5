"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each check is chosen so that a plausible mistake in the oracle fails it:
hand-derived routing and permutation cases (tests/golden/routing_hand.json),
brute-force top-k by explicit rank counting, closed-form gates, permutation
invariants, identity experts (combine must return x times the sum of kept
gates), a dense every-expert-then-mask formulation of the layer, the k=1 single
expert case against a textbook MLP written with torch.nn.functional, and
central finite differences for every gradient.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as orc
from synth import gen, workloads


@pytest.fixture(params=["numpy", "cpp"])
def impl(request):
    """The oracle under test: the numpy oracle or the C++ one; both must meet
    every pin that takes this fixture."""
    if request.param == "numpy":
        return orc
    from oracle import moe_oracle_cpp
    return moe_oracle_cpp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "routing_hand.json")


def _f(v):
    return float("-inf") if v == "-inf" else float(v)


# ---------------------------------------------------------------- golden
def test_golden_topk_cases(impl):
    cases = json.load(open(GOLDEN))["topk"]
    for c in cases:
        l = np.array([[_f(v) for v in row] for row in c["logits"]], dtype=np.float32)
        idx, g = impl.route_topk(l, c["k"])
        assert idx.tolist() == c["idx"], c["name"]
        np.testing.assert_allclose(g, np.array(c["gates"]), rtol=0, atol=1e-15, err_msg=c["name"])


def test_golden_permute_cases(impl):
    cases = json.load(open(GOLDEN))["permute"]
    for c in cases:
        idx = np.array(c["idx"], dtype=np.int32)
        p = impl.permute(idx, c["E"], c["capacity"])
        for key in ("counts_raw", "counts", "offsets", "row_of_slot", "slot_of_row"):
            assert p[key].tolist() == c[key], (c["name"], key)


# ---------------------------------------------------------------- top-k
def brute_force_topk(l: np.ndarray, k: int):
    """rank_e = #{e': l_e' > l_e} + #{e' < e: l_e' == l_e}; slot = rank."""
    T, E = l.shape
    idx = np.full((T, k), -1, dtype=np.int64)
    for t in range(T):
        for e in range(E):
            r = 0
            for e2 in range(E):
                if l[t, e2] > l[t, e] or (l[t, e2] == l[t, e] and e2 < e):
                    r += 1
            if r < k:
                idx[t, r] = e
    return idx


def _adversarial_logits(T, E, seed):
    rng = np.random.default_rng(seed)
    l = rng.standard_normal((T, E)).astype(np.float32)
    l[0] = 0.0                                  # all equal
    l[1, ::3] = 5.0                             # many maxima
    l[2] = -0.0; l[2, E // 2] = 0.0             # signed zeros
    l[3, : E // 2] = -np.inf                    # -inf columns
    l[4] = np.round(l[4])                       # coarse values, many ties
    l[5, E - 1] = np.float32(1e30)              # large value at the end
    return l


@pytest.mark.parametrize("E,k", [(8, 2), (8, 8), (64, 4), (128, 4), (256, 8), (5, 1)])
def test_topk_matches_brute_force(E, k, impl):
    l = _adversarial_logits(12, E, seed=E * 31 + k)
    idx, g = impl.route_topk(l, k)
    assert np.array_equal(idx, brute_force_topk(l, k))


@pytest.mark.parametrize("E,k", [(8, 2), (64, 4), (128, 4)])
def test_gates_closed_form(E, k, impl):
    l = gen.random_logits(64, E)
    idx, g = impl.route_topk(l, k)
    # softmax over all E, then renormalise over the selected set
    l64 = l.astype(np.float64)
    p = np.exp(l64 - l64.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    np.testing.assert_allclose(g, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12, atol=0)
    np.testing.assert_allclose(g.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.diff(g, axis=1) <= 0)  # slot order = descending gate


def test_random_routing_gates_are_softmax_over_the_k_drawn(impl):
    T, E, k = 256, 64, 4
    l = gen.random_routing_logits(T, E, k)
    assert np.all(np.isfinite(l).sum(axis=1) == k)
    idx, g = impl.route_topk(l, k)
    for t in range(T):
        fin = np.nonzero(np.isfinite(l[t]))[0]
        assert set(idx[t].tolist()) == set(fin.tolist())
        z = l[t, fin].astype(np.float64)
        sm = np.exp(z - z.max()) / np.exp(z - z.max()).sum()
        np.testing.assert_allclose(sorted(g[t]), sorted(sm), rtol=1e-12)


# ---------------------------------------------------------------- permutation
@pytest.mark.parametrize("T,E,k,cap", [(300, 8, 2, 0), (300, 8, 2, 40), (1000, 64, 4, 0),
                                       (1000, 64, 4, orc.capacity_of(1000, 4, 64)), (7, 4, 4, 1)])
def test_permutation_invariants(T, E, k, cap, impl):
    l = gen.random_logits(T, E)
    l[:, 0] += 1.0  # skew the load
    idx, _ = impl.route_topk(l, k)
    p = impl.permute(idx, E, cap)
    R = int(p["offsets"][-1])
    row = p["row_of_slot"]
    kept = row >= 0
    # bijection between kept slots and rows [0, R)
    assert sorted(row[kept].tolist()) == list(range(R))
    assert np.array_equal(p["slot_of_row"][row[kept]], np.nonzero(kept)[0])
    assert p["counts"].sum() == R == T * k - (~kept).sum()
    assert p["counts_raw"].sum() == T * k
    if cap > 0:
        assert np.all(p["counts"] <= cap)
    # each segment holds expert e's tokens, in strictly increasing token order
    for e in range(E):
        seg = p["slot_of_row"][p["offsets"][e]:p["offsets"][e + 1]]
        toks = seg // k
        assert np.all(idx.reshape(-1)[seg] == e)
        assert np.all(np.diff(toks) > 0)
        # dropped slots of e are exactly its latest tokens beyond the capacity
        all_toks = np.nonzero((idx == e).any(axis=1))[0]
        n_keep = len(all_toks) if cap <= 0 else min(cap, len(all_toks))
        assert np.array_equal(toks, all_toks[:n_keep])


# ---------------------------------------------------------------- layer pins
def _tiny_inputs(T, d, E, H, Hs, seed, learned=True):
    rng = np.random.default_rng(seed)
    inp = {
        "x": rng.standard_normal((T, d)),
        "W_g": 0.3 * rng.standard_normal((E, H, d)),
        "W_u": 0.3 * rng.standard_normal((E, H, d)),
        "W_d": 0.3 * rng.standard_normal((E, d, H)),
        "dY": rng.standard_normal((T, d)),
    }
    if learned:
        inp["W_r"] = 0.5 * rng.standard_normal((E, d))
    if Hs:
        inp["Ws_g"] = 0.3 * rng.standard_normal((Hs, d))
        inp["Ws_u"] = 0.3 * rng.standard_normal((Hs, d))
        inp["Ws_d"] = 0.3 * rng.standard_normal((d, Hs))
    return inp


@pytest.mark.parametrize("cap", [0, 3])
def test_identity_experts_return_x_times_sum_of_kept_gates(cap, impl):
    w = workloads.WORKLOADS["tiny"]
    inp = impl.inputs_to_f64(workloads.make_inputs(w))
    inp.pop("Ws_g", None)
    f = impl.layer_forward(inp, w.k, cap, expert_fn=lambda e, xr: xr)
    kept_gate_sum = (f["gates"] * f["kept"]).sum(axis=1)
    np.testing.assert_allclose(f["y"], inp["x"] * kept_gate_sum[:, None], rtol=1e-13, atol=1e-13)
    if cap == 0:
        np.testing.assert_allclose(kept_gate_sum, 1.0, atol=1e-12)
    else:
        assert (kept_gate_sum < 1.0 - 1e-9).any()


def dense_masked_layer(inp, k, cap):
    """Every expert on every token, then masked: y = s + sum_e m[t,e] G[t,e] f_e(x[t]).
    The mask comes from explicit rank counting, the gates from the full
    softmax renormalised over the mask, the capacity from a token-order count."""
    x = inp["x"]
    T, d = x.shape
    l = (x @ inp["W_r"].T).astype(np.float32).astype(np.float64)
    E = l.shape[1]
    sel_idx = brute_force_topk(l.astype(np.float32), k)
    mask = np.zeros((T, E), dtype=bool)
    for t in range(T):
        mask[t, sel_idx[t]] = True
    p = np.exp(l - l.max(axis=1, keepdims=True))
    G = np.where(mask, p, 0.0)
    G /= G.sum(axis=1, keepdims=True)
    keep = mask.copy()
    if cap > 0:
        seen = np.zeros(E, dtype=int)
        for t in range(T):
            for e in range(E):
                if mask[t, e]:
                    keep[t, e] = seen[e] < cap
                    seen[e] += 1
    y = np.zeros((T, d))
    for e in range(E):
        a = x @ inp["W_g"][e].T
        u = x @ inp["W_u"][e].T
        fe = (a / (1 + np.exp(-a)) * u) @ inp["W_d"][e].T
        y += (keep[:, e] * G[:, e])[:, None] * fe
    if "Ws_g" in inp:
        a = x @ inp["Ws_g"].T
        u = x @ inp["Ws_u"].T
        y += (a / (1 + np.exp(-a)) * u) @ inp["Ws_d"].T
    return y


@pytest.mark.parametrize("cap", [0, 5])
def test_routed_layer_equals_dense_masked_layer(cap, impl):
    inp = _tiny_inputs(T=24, d=16, E=6, H=12, Hs=8, seed=3)
    f = impl.layer_forward(inp, 2, cap)
    yd = dense_masked_layer(inp, 2, cap)
    np.testing.assert_allclose(f["y"], yd, rtol=1e-12, atol=1e-12)


def test_single_expert_k1_is_a_dense_swiglu_mlp(impl):
    inp = _tiny_inputs(T=10, d=16, E=1, H=24, Hs=8, seed=5)
    f = impl.layer_forward(inp, 1, 0)
    F = torch.nn.functional
    x = torch.tensor(inp["x"])

    def mlp(Wg, Wu, Wd):
        return F.linear(F.silu(F.linear(x, torch.tensor(Wg))) * F.linear(x, torch.tensor(Wu)), torch.tensor(Wd))

    y_ref = mlp(inp["W_g"][0], inp["W_u"][0], inp["W_d"][0]) + mlp(inp["Ws_g"], inp["Ws_u"], inp["Ws_d"])
    np.testing.assert_allclose(f["gates"], 1.0)
    np.testing.assert_allclose(f["y"], y_ref.numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- backward
def _loss(impl, inp, k, cap, **kw):
    f = impl.layer_forward(inp, k, cap, exact_router=True, **kw)
    return float((f["y"] * inp["dY"]).sum()), f


def _fd_setup(cap, seed0=11):
    # reseed until no top-k decision is within 1e-3 of flipping
    for seed in range(seed0, seed0 + 50):
        inp = _tiny_inputs(T=8, d=12, E=4, H=8, Hs=6, seed=seed)
        l = inp["x"] @ inp["W_r"].T
        s = -np.sort(-l, axis=1)
        if np.min(s[:, 1] - s[:, 2]) > 1e-3 and np.min(s[:, 0] - s[:, 1]) > 1e-3:
            return inp
    raise RuntimeError("no well-separated seed")


@pytest.mark.parametrize("cap", [0, 3])
def test_backward_matches_central_finite_differences(cap, impl):
    k = 2
    inp = _fd_setup(cap)
    _, f = _loss(impl, inp, k, cap)
    b = impl.layer_backward(inp, f)
    eps = 1e-6
    names = {"x": "dx", "W_r": "dW_r", "W_g": "dW_g", "W_u": "dW_u", "W_d": "dW_d",
             "Ws_g": "dWs_g", "Ws_u": "dWs_u", "Ws_d": "dWs_d"}
    for name, gname in names.items():
        P = inp[name]
        num = np.zeros_like(P)
        it = np.nditer(P, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = P[i]
            P[i] = old + eps
            lp, fp = _loss(impl, inp, k, cap)
            P[i] = old - eps
            lm, fm = _loss(impl, inp, k, cap)
            P[i] = old
            assert np.array_equal(fp["idx"], f["idx"]) and np.array_equal(fm["idx"], f["idx"])
            num[i] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(b[gname], num, rtol=1e-6, atol=1e-7, err_msg=gname)
    # gates treated as inputs
    G = f["gates"].copy()
    num = np.zeros_like(G)
    for i in np.ndindex(G.shape):
        Gp = G.copy(); Gp[i] += eps
        Gm = G.copy(); Gm[i] -= eps
        num[i] = (_loss(impl, inp, k, cap, gates=Gp)[0] - _loss(impl, inp, k, cap, gates=Gm)[0]) / (2 * eps)
    np.testing.assert_allclose(b["dgates"], num, rtol=1e-6, atol=1e-7)
    # logits treated as inputs
    L = f["logits"].copy()
    num = np.zeros_like(L)
    for i in np.ndindex(L.shape):
        Lp = L.copy(); Lp[i] += eps
        Lm = L.copy(); Lm[i] -= eps
        num[i] = (_loss(impl, inp, k, cap, logits=Lp)[0] - _loss(impl, inp, k, cap, logits=Lm)[0]) / (2 * eps)
    np.testing.assert_allclose(b["dlogits"], num, rtol=1e-6, atol=1e-7)


def test_swiglu_derivative_matches_torch_autograd():
    a = torch.linspace(-30, 30, 601, dtype=torch.float64, requires_grad=True)
    u = torch.linspace(-2, 3, 601, dtype=torch.float64)
    h = torch.nn.functional.silu(a) * u
    h.sum().backward()
    sg = orc.sigmoid(a.detach().numpy())
    da = u.numpy() * sg * (1 + a.detach().numpy() * (1 - sg))
    np.testing.assert_allclose(da, a.grad.numpy(), rtol=1e-12, atol=1e-14)


def test_capacity_formula():
    assert orc.capacity_of(8192, 4, 64) == 640          # 1.25 * 8192 * 4 / 64 exactly
    assert orc.capacity_of(10, 1, 3) == math.ceil(1.25 * 10 / 3)
    assert workloads.WORKLOADS["tiny64e_zipf_cap125"].capacity == 640
    # other factors, as the fractions they denote: ceil(0.25 * 700 * 4 / 16) =
    # ceil(43.75) = 44; an exact multiple does not round up
    assert workloads.custom("c", T=700, d=256, E=16, k=4, H=256, Hs=0, capacity_factor=0.25).capacity == 44
    assert workloads.custom("c", T=64, d=256, E=16, k=4, H=256, Hs=0, capacity_factor=0.5).capacity == 8
    assert workloads.custom("c", T=64, d=256, E=16, k=4, H=256, Hs=0).capacity == 0


# ---------------------------------------------------------------- balance loss
BALANCE_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "balance_loss_hand.json")


def test_golden_balance_loss_cases():
    for c in json.load(open(BALANCE_GOLDEN))["cases"]:
        l = np.array([[_f(v) for v in row] for row in c["logits"]], dtype=np.float64)
        L, f, P, dl = orc.balance_loss(l, np.array(c["idx"]), c["E"], c["alpha"])
        assert abs(L - c["loss"]) < 1e-12, c["name"]
        np.testing.assert_allclose(f, c["f"], rtol=0, atol=1e-15, err_msg=c["name"])
        np.testing.assert_allclose(P, c["P"], rtol=0, atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(dl, np.array(c["dl"], dtype=np.float64), rtol=0, atol=1e-12, err_msg=c["name"])


@pytest.mark.parametrize("E,k", [(5, 2), (8, 3), (64, 4)])
def test_balance_loss_gradient_matches_finite_differences(E, k):
    """The assignments are held fixed (they are piecewise constant in the
    logits); a central difference of the loss itself checks dL/dl."""
    rng = np.random.default_rng(E * 10 + k)
    T = 7
    l = rng.normal(size=(T, E))
    idx, _ = orc.route_topk(l.astype(np.float32), k)
    alpha = 0.05
    L0, f, P, dl = orc.balance_loss(l, idx, E, alpha)
    eps = 1e-6
    for t, j in [(0, 0), (3, E - 1), (6, E // 2), (2, 1)]:
        lp, lm = l.copy(), l.copy()
        lp[t, j] += eps
        lm[t, j] -= eps
        num = (orc.balance_loss(lp, idx, E, alpha)[0] - orc.balance_loss(lm, idx, E, alpha)[0]) / (2 * eps)
        assert abs(num - dl[t, j]) <= 1e-8 + 1e-6 * abs(dl[t, j]), (t, j, num, dl[t, j])


def test_balance_loss_invariants():
    """f and P are distributions; the gradient of every token sums to zero
    (softmax); perfect balance gives alpha; the loss is linear in alpha."""
    rng = np.random.default_rng(3)
    T, E, k = 50, 16, 4
    l = rng.normal(size=(T, E)) * 2.0
    idx, _ = orc.route_topk(l.astype(np.float32), k)
    L, f, P, dl = orc.balance_loss(l, idx, E, 0.2)
    assert abs(f.sum() - 1) < 1e-12 and abs(P.sum() - 1) < 1e-12
    np.testing.assert_allclose(dl.sum(axis=1), 0.0, atol=1e-15)
    assert abs(orc.balance_loss(l, idx, E, 0.5)[0] - 2.5 * L) < 1e-12
    # balanced assignments and equal logits: L = alpha exactly
    idx_b = np.array([[(t * k + s) % E for s in range(k)] for t in range(E)])
    assert abs(orc.balance_loss(np.zeros((E, E)), idx_b, E, 0.3)[0] - 0.3) < 1e-12


# ---------------------------------------------------------------- bf16 decode
# Hand-written bf16 bit patterns and the values the format definition gives
# them (sign | 8-bit exponent, bias 127 | 7-bit mantissa; exponent 0 =
# subnormal with scale 2^-126).
BF16_KNOWN = [
    (0x0000, 0.0), (0x8000, -0.0), (0x3F80, 1.0), (0xC040, -3.0), (0x4049, 3.140625),
    (0x3C00, 2.0 ** -7), (0x0001, 2.0 ** -133), (0x007F, 127 * 2.0 ** -133), (0x0080, 2.0 ** -126),
    (0x7F7F, 255 * 2.0 ** 120), (0xFF7F, -255 * 2.0 ** 120), (0x7F80, math.inf), (0xFF80, -math.inf),
]


def test_bf16_to_f64_known_values(impl):
    bits = np.array([b for b, _ in BF16_KNOWN], dtype=np.uint16)
    got = impl.bf16_to_f64(bits)
    assert got.dtype == np.float64
    for (b, want), g in zip(BF16_KNOWN, got):
        assert g == want and math.copysign(1.0, g) == math.copysign(1.0, want), (hex(b), g, want)
    # a 2-D array keeps its shape
    assert impl.bf16_to_f64(bits[:12].reshape(3, 4)).shape == (3, 4)


# ---------------------------------------------------------------- router bias
BIAS_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "router_bias_hand.json")


def _bias_case(c):
    # the hand-written bit patterns decoded by the numpy oracle (pinned by
    # test_bf16_to_f64_known_values)
    x = orc.bf16_to_f64(np.array([[int(h, 16) for h in c["x_bits"]]], dtype=np.uint16))
    W_r = orc.bf16_to_f64(np.array([[int(h, 16) for h in row] for row in c["W_r_bits"]], dtype=np.uint16))
    bias = np.array(c["bias"], dtype=np.float32)
    return x, W_r, bias


def _k2_gates(c):
    if "gates" in c["k2"]:
        return np.array([c["k2"]["gates"]])
    z = math.exp(-1.0 / 8.0)  # the closed form the second case states
    return np.array([[1.0 / (1.0 + z), z / (1.0 + z)]])


def check_router_bias_golden(layer_forward=None, router_logits=None, impl=orc):
    """The golden cases through the oracle's router and through its whole
    forward (identity experts), so that the bias is pinned where the layer
    applies it: in the fp32 logits that both the selection and the gates
    use."""
    layer_forward = layer_forward or impl.layer_forward
    router_logits = router_logits or impl.router_logits
    for c in json.load(open(BIAS_GOLDEN))["cases"]:
        x, W_r, bias = _bias_case(c)
        l = router_logits(x, W_r, bias)
        assert l.dtype == np.float32, c["name"]
        assert l[0].tolist() == c["logits"], (c["name"], l[0].tolist())
        for k, key in ((1, "k1"), (2, "k2")):
            f = layer_forward({"x": x, "W_r": W_r, "bias": bias}, k, 0, expert_fn=lambda e, xr: xr)
            assert f["idx"].tolist() == [c[key]["idx"]], (c["name"], k, f["idx"].tolist())
            want = np.array([c[key]["gates"]]) if k == 1 else _k2_gates(c)
            np.testing.assert_allclose(f["gates"], want, rtol=0, atol=1e-15, err_msg=f"{c['name']} k={k}")


def test_router_bias_golden(impl):
    check_router_bias_golden(impl=impl)


def test_router_bias_moves_selection_and_gates(impl):
    """A large bias on one expert puts it first for every token, and the gates
    are the softmax of the biased logits over the selection."""
    T, d, E, k = 64, 32, 8, 2
    x = impl.bf16_to_f64(gen.normal_bf16(501, (T, d)))
    W_r = impl.bf16_to_f64(gen.normal_bf16(502, (E, d), std=0.02))
    bias = np.zeros(E, dtype=np.float32)
    bias[5] = 30.0
    f = impl.layer_forward({"x": x, "W_r": W_r, "bias": bias}, k, 0, expert_fn=lambda e, xr: xr)
    assert np.all(f["idx"][:, 0] == 5)
    l = (x @ W_r.T).astype(np.float32) + bias  # fp32 product, then the fp32 add
    sel = np.take_along_axis(l.astype(np.float64), f["idx"].astype(np.int64), axis=1)
    g = np.exp(sel - sel[:, :1])
    np.testing.assert_allclose(f["gates"], g / g.sum(axis=1, keepdims=True), rtol=1e-12)
    assert np.all(f["gates"][:, 0] > 0.999)  # the gap of ~30 is in the gates too


def test_router_bias_pins_catch_planted_mistakes():
    """Each plausible mistake in the bias branch, planted in a copy of the
    oracle's router on the CPU, fails the golden check."""
    def fp64_add(x, W_r, bias=None):  # bias added before the fp32 rounding
        return (x @ W_r.T + np.asarray(bias, dtype=np.float64)[None, :]).astype(np.float32)

    def sign_flip(x, W_r, bias=None):
        return (x @ W_r.T).astype(np.float32) - np.asarray(bias, dtype=np.float32)[None, :]

    def no_bias(x, W_r, bias=None):
        return (x @ W_r.T).astype(np.float32)

    def selection_only(inp, k, cap, expert_fn=None):  # gates from the unbiased logits
        f = orc.layer_forward(inp, k, cap, expert_fn=expert_fn)
        l0 = (inp["x"] @ inp["W_r"].T).astype(np.float32).astype(np.float64)
        sel = np.take_along_axis(l0, f["idx"].astype(np.int64), axis=1)
        g = np.exp(sel - sel.max(axis=1, keepdims=True))
        return orc.layer_forward(inp, k, cap, expert_fn=expert_fn, gates=g / g.sum(axis=1, keepdims=True))

    for bad in (fp64_add, sign_flip, no_bias):
        saved = orc.router_logits
        orc.router_logits = bad
        try:
            with pytest.raises(AssertionError):
                check_router_bias_golden()
        finally:
            orc.router_logits = saved
    with pytest.raises(AssertionError):
        check_router_bias_golden(layer_forward=selection_only)
