"""Helpers shared by the GPU tests: upload of the seeded inputs, the parity
tolerance, and the routing near-tie analysis."""
from __future__ import annotations

import math

import numpy as np
import torch

# Floating-point parity bar of the layer: elementwise |gpu - ref| <= ATOL + RTOL*|ref|
# and relative Frobenius error <= FRO per tensor.
ATOL = 1e-2
RTOL = 2e-2
FRO = 5e-3


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def upload(inp: dict) -> dict:
    out = {}
    for key, v in inp.items():
        if v is None:
            continue
        if key in ("bias", "logits_in"):
            out[key] = dev_f32(v)
        else:
            out[key] = dev_bf16(v)
    return out


MARGINS = {}  # name -> (max err/bound, relative Frobenius), of the last comparison


def assert_close(name, gpu: np.ndarray, ref: np.ndarray, atol=ATOL, rtol=RTOL, fro=FRO, allow=None):
    """allow: an optional per-element absolute allowance added to the bound
    (a rounding bound derived from the arithmetic, for shapes beyond the
    layer configurations the bar is stated for)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values"
    err = np.abs(gpu - ref)
    bound = atol + rtol * np.abs(ref)
    if allow is not None:
        bound = bound + np.broadcast_to(np.asarray(allow, dtype=np.float64), bound.shape)
    bad = err > bound
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(gpu - ref) / nref if nref > 0 else np.linalg.norm(gpu)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = float(np.max(np.where(bound > 0, err / np.where(bound > 0, bound, 1), np.where(err > 0, np.inf, 0))))
    MARGINS[name] = (ratio, float(rel))
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} elements out of tolerance; worst at {i}: "
                             f"gpu {gpu[i]!r} ref {ref[i]!r}; rel fro {rel:.3e}")
    assert rel <= fro, f"{name}: relative Frobenius error {rel:.3e} > {fro}"
    return rel


_assert_close = assert_close  # for compare_layer, whose local wrapper shadows the name


def near_tie_tokens(logits: np.ndarray, k: int, delta: float) -> np.ndarray:
    """Tokens whose top-k SET could change under a perturbation of the logits
    by up to delta (gap between the k-th and (k+1)-th largest < 2*delta)."""
    E = logits.shape[1]
    if k >= E:
        return np.zeros(logits.shape[0], dtype=bool)
    s = -np.sort(-logits.astype(np.float64), axis=1)
    return (s[:, k - 1] - s[:, k]) < 2 * delta


def valid_topk_within(logits_row: np.ndarray, chosen, delta: float) -> bool:
    """True if `chosen` is a top-k set of logits_row for some perturbation of
    at most delta per logit."""
    chosen = set(int(c) for c in chosen)
    l = logits_row.astype(np.float64)
    lo_in = min(l[c] for c in chosen)
    others = [l[e] for e in range(len(l)) if e not in chosen]
    return not others or max(others) <= lo_in + 2 * delta


def routing_disagreements(gpu_idx: np.ndarray, ref_idx: np.ndarray, ref_logits: np.ndarray, k: int,
                          delta: float) -> np.ndarray:
    """Tokens whose GPU top-k (as an ordered list) differs from the oracle's.
    Each such token must sit at a near tie of the oracle's logits (a gap
    below 2*delta, delta = the fp32-vs-fp64 router rounding allowance) and the
    GPU's set must be a valid top-k within delta.  Returns the mask."""
    diff = ~(gpu_idx == ref_idx).all(axis=1)
    if not diff.any():
        return diff
    l = ref_logits.astype(np.float64)
    s = -np.sort(-l, axis=1)
    gaps = np.abs(np.diff(s[:, : min(k + 1, l.shape[1])], axis=1)).min(axis=1)
    for t in np.nonzero(diff)[0]:
        assert gaps[t] < 2 * delta, f"token {t}: routing differs without a near tie (min gap {gaps[t]:.3e})"
        assert valid_topk_within(l[t], gpu_idx[t], delta), f"token {t}: GPU top-k is not a valid selection"
    return diff


LOGIT_TOL = 1e-4


class ParityInfo(UserWarning):
    """Informational note of a parity test (shown in pytest's warnings
    summary): e.g. how many tokens the fp32 router logits route differently
    from the fp64-router oracle at near ties."""


def oracle_reference(w, inp, layer, f64=None, impl=None):
    """The oracle's forward and backward for a finished GPU layer run.

    Learned routing: the GPU's fp32 logits are first checked against the
    oracle's router (elementwise within LOGIT_TOL), and the GPU's top-k against
    the oracle's selection on its own logits (a token may differ only at a
    near tie, and the GPU's set must then be a valid top-k within the router
    rounding allowance).  The oracle then runs the whole layer on the GPU's
    logits, so that routing, permutation, gates and every downstream value are
    compared on the same fp32 logits, with no token or expert left out.
    impl: the oracle module (default the numpy one; oracle.moe_oracle_cpp
    has the same interface).  Returns (f64 inputs, forward dict, backward
    dict, number of near-tie tokens)."""
    import warnings
    from oracle import moe_oracle
    orc = impl or moe_oracle
    if f64 is None:
        f64 = orc.inputs_to_f64(inp)
    flips = 0
    logits = None
    if w.routing == "learned":
        gl = layer.logits.cpu().numpy()
        ol = orc.router_logits(f64["x"], f64["W_r"], f64.get("bias"))
        np.testing.assert_allclose(gl, ol, rtol=0, atol=LOGIT_TOL)
        delta = max(float(np.abs(gl.astype(np.float64) - ol).max()), 1e-7) * 4
        oidx, _ = orc.route_topk(ol, w.k)
        diff = routing_disagreements(layer.idx.cpu().numpy(), oidx, ol, w.k, delta)
        flips = int(diff.sum())
        assert flips <= max(1, w.T // 100), f"{flips} near-tie flips"
        if flips:
            warnings.warn(ParityInfo(f"{w.name}: {flips} of {w.T} tokens route differently on the GPU's fp32 "
                                     f"logits than on the oracle's (near ties); all routing checks ran bit-exact "
                                     f"on the GPU's logits"))
        logits = gl
    ref = orc.layer_forward(f64, w.k, w.capacity, logits=logits)
    refb = orc.layer_backward(f64, ref)
    return f64, ref, refb, flips


def compare_layer(w, inp, layer, ref, refb, allow=None):
    """Compares a finished MoELayer forward+backward with the oracle's
    (`oracle_reference`: the oracle run on the same fp32 logits).  Top-k
    indices, counts, offsets, both row maps, x_perm and dY_perm bit-exact;
    every floating output and gradient within the layer tolerance, every
    token and every expert.  A fused layer (the permutation inside the GEMMs'
    loads, the combine inside the shared down projection) has no x_perm,
    dY_perm or s, and holds the expert outputs by slot.  allow: optional
    per-element allowances by tensor name (assert_close)."""
    import torch
    MARGINS.clear()
    k = w.k
    allow = allow or {}

    def assert_close(name, gpu, ref_, **kw):
        return _assert_close(name, gpu, ref_, allow=allow.get(name), **kw)

    # routing and permutation: bit-exact
    assert np.array_equal(layer.idx.cpu().numpy(), ref["idx"]), "topk_idx"
    for key in ("counts_raw", "counts", "offsets", "row_of_slot"):
        assert np.array_equal(getattr(layer, key).cpu().numpy(), ref[key]), key
    R = int(ref["offsets"][-1])
    assert np.array_equal(layer.slot_of_row.cpu().numpy()[:R], ref["slot_of_row"]), "slot_of_row"
    fused = getattr(layer, "fused", False)
    if not fused:
        xp = layer.x_perm.view(torch.int16).cpu().numpy().view(np.uint16)[:R]
        assert np.array_equal(xp, inp["x"][ref["slot_of_row"] // k]), "x_perm"
        dyp = layer.dY_perm.view(torch.int16).cpu().numpy().view(np.uint16)[:R]
        assert np.array_equal(dyp, inp["dY"][ref["slot_of_row"] // k]), "dY_perm"
    # gates: fp32 expf on the GPU against float64
    np.testing.assert_allclose(layer.gates.cpu().numpy(), ref["gates"], rtol=1e-5, atol=1e-6)

    # forward values, per kept row and per token
    if layer.au is not None:
        assert_close("a", host_f64(layer.au[:R, :w.H]), ref["a"])
        assert_close("u", host_f64(layer.au[:R, w.H:]), ref["u"])
    assert_close("h", host_f64(layer.h[:R]), ref["h"])
    if fused:
        # expert outputs stored by slot: row r's output at slot_of_row[r]
        slots = torch.from_numpy(ref["slot_of_row"].astype(np.int64)).to(layer.o_perm.device)
        assert_close("o_slot", host_f64(layer.o_perm[slots]), ref["o"])
    else:
        assert_close("o_perm", host_f64(layer.o_perm[:R]), ref["o"])
    if w.Hs and not fused:
        assert_close("s", host_f64(layer.s), ref["s"])
    assert_close("y", host_f64(layer.y), ref["y"])

    # backward; the stored fp16 input-gradient terms are the values divided by
    # 2^e, e = floor(log2 max|dY|), when the layer keeps a gradient scale word
    # (which must hold max|dY|'s bf16 magnitude pattern)
    up = 1.0
    if getattr(layer, "dx_scale", None) is not None:
        m = int((inp["dY"].astype(np.uint32) & 0x7FFF).max())
        assert (int(layer.dx_scale.item()) & 0xFFFFFFFF) == m, "gradient scale word"
        amax = float(np.array([m << 16], dtype=np.uint32).view(np.float32)[0])
        if 0.0 < amax < np.inf:
            up = 2.0 ** math.floor(math.log2(amax))
    assert_close("dx_perm", host_f64(layer.dx_perm[:R]) * up, refb["dx_perm"])
    assert_close("dgates", layer.dgates.cpu().numpy(), refb["dgates"])
    assert_close("dW_d", host_f64(layer.dW_d), refb["dW_d"])
    assert_close("dW_g", host_f64(layer.dW_g), refb["dW_g"])
    assert_close("dW_u", host_f64(layer.dW_u), refb["dW_u"])
    if w.Hs:
        assert_close("dx_s", host_f64(layer.dx_s) * up, refb["dx_s"])
        assert_close("dWs_d", host_f64(layer.dWs_d), refb["dWs_d"])
        assert_close("dWs_g", host_f64(layer.dWs_g), refb["dWs_g"])
        assert_close("dWs_u", host_f64(layer.dWs_u), refb["dWs_u"])
    assert_close("dlogits", layer.dlogits.cpu().numpy(), refb["dlogits"])
    if w.routing == "learned":
        assert_close("dW_r", layer.dW_r.cpu().numpy(), refb["dW_r"])
    assert_close("dx", host_f64(layer.dx), refb["dx"])
    worst = ", ".join(f"{n} {r:.2f}/{f:.1e}" for n, (r, f) in sorted(MARGINS.items(), key=lambda kv: -kv[1][0]))
    print(f"[margins: max err/bound / rel fro] {worst}")
