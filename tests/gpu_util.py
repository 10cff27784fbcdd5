"""Helpers shared by the GPU tests: upload of the seeded inputs, the parity
tolerance, and the routing near-tie analysis."""
from __future__ import annotations

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


MARGINS = {}  # name -> (max err/(atol + rtol|ref|), relative Frobenius), of the last comparison


def assert_close(name, gpu: np.ndarray, ref: np.ndarray, atol=ATOL, rtol=RTOL, fro=FRO):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values"
    err = np.abs(gpu - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(gpu - ref) / nref if nref > 0 else np.linalg.norm(gpu)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = float(np.max(np.where(bound > 0, err / np.where(bound > 0, bound, 1), np.where(err > 0, np.inf, 0))))
    MARGINS[name] = (ratio, float(rel))
    if bad.any():
        i = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(ref))), err.shape)
        raise AssertionError(f"{name}: {bad.sum()} of {bad.size} elements out of tolerance; worst at {i}: "
                             f"gpu {gpu[i]!r} ref {ref[i]!r}; rel fro {rel:.3e}")
    assert rel <= fro, f"{name}: relative Frobenius error {rel:.3e} > {fro}"
    return rel


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


def experts_touched(tokens_mask: np.ndarray, *idx_arrays) -> np.ndarray:
    """Experts selected by any of the masked tokens in any of the idx arrays."""
    out = set()
    for idx in idx_arrays:
        out.update(np.unique(idx[tokens_mask]).tolist())
    return np.array(sorted(out), dtype=np.int64)


LOGIT_TOL = 1e-4


def compare_layer(w, inp, layer, ref, refb):
    """Compares a finished MoELayer forward+backward with the oracle's
    (layer_forward / layer_backward on the same inputs).  Routing and
    permutation bit-exact (apart from legitimate near-tie flips under learned
    routing, which are excluded from the per-token and per-expert checks),
    floating outputs within the layer tolerance."""
    import torch
    MARGINS.clear()
    T, k = w.T, w.k

    gidx = layer.idx.cpu().numpy()
    diff = np.zeros(T, dtype=bool)
    if w.routing == "learned":
        gl = layer.logits.cpu().numpy()
        np.testing.assert_allclose(gl, ref["logits"], rtol=0, atol=LOGIT_TOL)
        delta = max(float(np.abs(gl.astype(np.float64) - ref["logits"]).max()), 1e-7) * 4
        diff = routing_disagreements(gidx, ref["idx"], ref["logits"], k, delta)
        assert diff.sum() <= max(1, T // 100)
    else:
        assert np.array_equal(gidx, ref["idx"])
    keep = ~diff
    skip_e = experts_touched(diff, gidx, ref["idx"])
    keep_e = np.setdiff1d(np.arange(w.E), skip_e)
    if w.capacity > 0 and diff.any():
        # a flipped token shifts the token-order ranks (and so the drops) of
        # later tokens in the experts it touches
        keep &= ~np.isin(ref["idx"], skip_e).any(axis=1) & ~np.isin(gidx, skip_e).any(axis=1)
    if not diff.any():
        # routing and permutation: bit-exact
        for key in ("counts_raw", "counts", "offsets", "row_of_slot"):
            assert np.array_equal(getattr(layer, key).cpu().numpy(), ref[key]), key
        R = int(ref["offsets"][-1])
        assert np.array_equal(layer.slot_of_row.cpu().numpy()[:R], ref["slot_of_row"])
        assert_close("x_perm", host_f64(layer.x_perm[:R]), ref["x_perm"], atol=0, rtol=0, fro=0)
        assert_close("h", host_f64(layer.h[:R]), ref["h"])
        assert_close("a", host_f64(layer.au[:R, :w.H]), ref["a"])
        assert_close("u", host_f64(layer.au[:R, w.H:]), ref["u"])
        assert_close("o_perm", host_f64(layer.o_perm[:R]), ref["o"])
        dyp = layer.dY_perm.view(torch.int16).cpu().numpy().view(np.uint16)[:R]
        assert np.array_equal(dyp, inp["dY"][ref["slot_of_row"] // k])
        assert_close("dx_perm", host_f64(layer.dx_perm[:R]), refb["dx_perm"])
    np.testing.assert_allclose(layer.gates.cpu().numpy()[keep], ref["gates"][keep], rtol=1e-5, atol=1e-6)

    # forward values
    if w.Hs:
        assert_close("s", host_f64(layer.s), ref["s"])
    assert_close("y", host_f64(layer.y)[keep], ref["y"][keep])

    # backward
    assert_close("dgates", layer.dgates.cpu().numpy()[keep], refb["dgates"][keep])
    assert_close("dW_d", host_f64(layer.dW_d)[keep_e], refb["dW_d"][keep_e])
    assert_close("dW_g", host_f64(layer.dW_g)[keep_e], refb["dW_g"][keep_e])
    assert_close("dW_u", host_f64(layer.dW_u)[keep_e], refb["dW_u"][keep_e])
    if w.Hs:
        assert_close("dx_s", host_f64(layer.dx_s), refb["dx_s"])
        assert_close("dWs_d", host_f64(layer.dWs_d), refb["dWs_d"])
        assert_close("dWs_g", host_f64(layer.dWs_g), refb["dWs_g"])
        assert_close("dWs_u", host_f64(layer.dWs_u), refb["dWs_u"])
    assert_close("dlogits", layer.dlogits.cpu().numpy()[keep], refb["dlogits"][keep])
    if w.routing == "learned":
        assert_close("dW_r", layer.dW_r.cpu().numpy()[keep_e], refb["dW_r"][keep_e])
    assert_close("dx", host_f64(layer.dx)[keep], refb["dx"][keep])
    worst = ", ".join(f"{n} {r:.2f}/{f:.1e}" for n, (r, f) in sorted(MARGINS.items(), key=lambda kv: -kv[1][0]))
    print(f"[margins: max err/bound / rel fro] {worst}")
    return int(diff.sum())
