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


def assert_close(name, gpu: np.ndarray, ref: np.ndarray, atol=ATOL, rtol=RTOL, fro=FRO):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (name, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values"
    err = np.abs(gpu - ref)
    bad = err > atol + rtol * np.abs(ref)
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(gpu - ref) / nref if nref > 0 else np.linalg.norm(gpu)
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
