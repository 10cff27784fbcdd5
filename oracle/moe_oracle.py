"""CPU oracle of the MoE layer with top-k routing and one shared expert.

TEST INFRASTRUCTURE ONLY.  Only the tests, `__graft_entry__.smoke()` and the
bench's CPU-baseline / reference leg may import this module.  The CUDA library
never calls it, and it shares no code with the CUDA path.

Plain, slow and obviously correct: every quantity is computed from its
definition in float64 (numpy), on float64 copies of the bf16 inputs.  No
intermediate is rounded to bf16.  Matrix products (`@`) are the only library
primitive used.  No blocking, fusion or reordering beyond the definitions.

What the layer computes (the sources are the Olmo-core DDP MoE pages: the
"Olmo-core DDP MoE examples" README, "Production throughput runs" (top-4
routing, one shared expert, random vs learned routing) and "Interpreting the
eight-layer DDP vs FSDP comparison" (capacity factor, router, shared-branch
mixing); "Olmo-core 3 Opens Large MoE Training", "Technical Deep Dive" (experts
stay resident, tokens are routed to them); "Scaling Trillion-Parameter Models:
The Architecture of Olmo-core 3", "Code Snippet" (a per-token expert-selection
step)).  The pages give no formulas for the layer; the definitions below are
the plainest reading of the problem they describe: softmax routing in fp32,
the top-k gates renormalised to sum to 1, the per-expert stable permutation,
a SwiGLU expert MLP without biases, the shared expert added with weight 1, and
capacity overflow dropped in token-index order without renormalising.

  router    l[t,e] = fp32( sum_c x[t,c] W_r[e,c] ) + b[e]          (fp32 add)
  top-k     S(t) = the k experts first in the order (l desc, e asc);
            slot s = position in that order (ties -> lower expert index)
  gates     g[t,s] = exp(l_s - m) / sum_{j in S} exp(l_j - m)       (= softmax
            over all E renormalised over S)
  rank      rank(t,s) = #{t' < t : idx[t,s] in S(t')}
  capacity  kept iff C <= 0 (dropless) or rank < C; dropped gates are not
            renormalised
  permute   counts_raw[e], counts[e] = #kept, offsets = exclusive prefix sum,
            row(t,s) = offsets[e] + rank, x_perm[row] = x[t]
  expert    a = x W_g[e]^T, u = x W_u[e]^T, h = silu(a) * u, o = h W_d[e]^T
  shared    s[t] = same SwiGLU with the shared weights, added with weight 1
  combine   y[t] = s[t] + sum_{s kept} g[t,s] o[row(t,s)]

Backward (upstream dY):
  dO[row] = g dY[t];  dg[t,s] = <dY[t], o[row]> (0 if dropped)
  dh = dO W_d;  dW_d = dO^T h;  da = dh u sig(a)(1 + a(1 - sig(a)));
  du = dh silu(a);  dx_e = da W_g + du W_u;  dW_g = da^T x_e;  dW_u = du^T x_e
  dl[t,e_s] = g_s (dg_s - sum_j g_j dg_j), 0 for experts outside S(t)
  dW_r = dl^T x;   dx[t] = sum_s dx_e[row(t,s)] + dx_shared[t] + dl[t] W_r
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# conversions of the stored inputs
# --------------------------------------------------------------------------
def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values (exact)."""
    return (np.asarray(b).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def sigmoid(a):
    return 1.0 / (1.0 + np.exp(-a))


def silu(a):
    return a * sigmoid(a)


# --------------------------------------------------------------------------
# routing
# --------------------------------------------------------------------------
def router_logits(x: np.ndarray, W_r: np.ndarray, bias=None) -> np.ndarray:
    """l = fp32(x W_r^T) + bias, the fp32 add done in fp32.
    x [T,d] float64, W_r [E,d] float64, bias [E] float32 or None."""
    l = (x @ W_r.T).astype(np.float32)
    if bias is not None:
        l = l + np.asarray(bias, dtype=np.float32)[None, :]
    return l


def route_topk(logits: np.ndarray, k: int):
    """Top-k selection and renormalised gates from fp32 logits [T,E].

    Returns idx [T,k] int32 (slot order: logit descending, ties to the lower
    expert index) and gates [T,k] float64.  The comparison is made on the
    logits as given (fp32 for the layer; fp64 only in finite-difference
    checks)."""
    l = np.asarray(logits)
    if l.dtype != np.float64:
        l = l.astype(np.float32)
    T, E = l.shape
    # stable sort of the negated logits: descending value, equal values keep
    # ascending expert index; -0.0 and +0.0 compare equal.
    order = np.argsort(-l, axis=1, kind="stable")
    idx = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(l, idx.astype(np.int64), axis=1).astype(np.float64)
    m = sel[:, :1]
    with np.errstate(invalid="ignore"):
        ex = np.exp(sel - m)
    ex = np.where(np.isnan(ex), 0.0, ex)  # -inf - (-inf) only if all k are -inf
    den = ex.sum(axis=1, keepdims=True)
    gates = ex / den
    return idx, gates


def capacity_of(T: int, k: int, E: int, factor_num: int = 5, factor_den: int = 4) -> int:
    """C = ceil(factor * T * k / E), exact in integers (factor = num/den)."""
    return (factor_num * T * k + factor_den * E - 1) // (factor_den * E)


def permute(idx: np.ndarray, E: int, capacity: int = 0):
    """Histogram, capacity drop, exclusive prefix sum and stable scatter map.

    Returns dict with counts_raw [E], counts [E], offsets [E+1], rank [T,k],
    kept [T,k] bool, row_of_slot [T*k] (-1 = dropped), slot_of_row [R]."""
    T, k = idx.shape
    rank = np.zeros((T, k), dtype=np.int64)
    counts_raw = np.zeros(E, dtype=np.int64)
    for e in range(E):
        ts, ss = np.nonzero(idx == e)  # row-major: increasing token index
        rank[ts, ss] = np.arange(len(ts))
        counts_raw[e] = len(ts)
    if capacity > 0:
        kept = rank < capacity
        counts = np.minimum(counts_raw, capacity)
    else:
        kept = np.ones((T, k), dtype=bool)
        counts = counts_raw.copy()
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    row = np.where(kept, offsets[idx] + rank, -1)
    R = int(offsets[E])
    slot_of_row = np.full(R, -1, dtype=np.int64)
    flat = row.reshape(-1)
    slots = np.nonzero(flat >= 0)[0]
    slot_of_row[flat[slots]] = slots
    return {
        "counts_raw": counts_raw, "counts": counts, "offsets": offsets,
        "rank": rank, "kept": kept, "row_of_slot": flat.copy(), "slot_of_row": slot_of_row,
    }


# --------------------------------------------------------------------------
# expert MLP (SwiGLU)
# --------------------------------------------------------------------------
def swiglu_fwd(xr: np.ndarray, Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray):
    """xr [n,d]; Wg, Wu [H,d]; Wd [d,H]  ->  (a, u, h, o)."""
    a = xr @ Wg.T
    u = xr @ Wu.T
    h = silu(a) * u
    o = h @ Wd.T
    return a, u, h, o


def swiglu_bwd(xr, Wg, Wu, Wd, a, u, h, dO):
    """Gradients of o = (silu(x Wg^T) * (x Wu^T)) Wd^T.  Returns
    (dx, dWg, dWu, dWd, da, du)."""
    dh = dO @ Wd
    dWd = dO.T @ h
    sg = sigmoid(a)
    da = dh * u * sg * (1.0 + a * (1.0 - sg))
    du = dh * silu(a)
    dx = da @ Wg + du @ Wu
    dWg = da.T @ xr
    dWu = du.T @ xr
    return dx, dWg, dWu, dWd, da, du


# --------------------------------------------------------------------------
# combine / unpermute steps and their backward
# --------------------------------------------------------------------------
def combine(o, s, gates, row_of_slot, T, k):
    """y[t] = s[t] + sum_{s kept} g[t,s] o[row(t,s)]  (s may be None)."""
    d = o.shape[1]
    y = np.zeros((T, d)) if s is None else np.array(s, dtype=np.float64, copy=True)
    row = np.asarray(row_of_slot).reshape(T, k)
    for s_ in range(k):
        m = row[:, s_] >= 0
        y[m] += gates[m, s_:s_ + 1] * o[row[m, s_]]
    return y


def combine_bwd(dY, o, gates, row_of_slot, T, k):
    """dO[row] = g dY[t]; dg[t,s] = <dY[t], o[row]> (0 for dropped slots)."""
    d = dY.shape[1]
    row = np.asarray(row_of_slot).reshape(T, k)
    R = o.shape[0]
    dO = np.zeros((R, d))
    dg = np.zeros((T, k))
    for s_ in range(k):
        m = row[:, s_] >= 0
        dO[row[m, s_]] = gates[m, s_:s_ + 1] * dY[m]
        dg[m, s_] = np.einsum("tc,tc->t", dY[m], o[row[m, s_]])
    return dO, dg


def topk_bwd(gates, idx, dg, E):
    """Softmax-over-the-selected Jacobian: dl[t, idx[t,s]] = g_s (dg_s -
    sum_j g_j dg_j), zero for experts outside the selection."""
    T, k = idx.shape
    dl = np.zeros((T, E))
    sgd = (gates * dg).sum(axis=1, keepdims=True)
    np.put_along_axis(dl, np.asarray(idx).astype(np.int64), gates * (dg - sgd), axis=1)
    return dl


def permute_bwd(dx_perm, dx_s, row_of_slot, T, k, dl=None, W_r=None):
    """dx[t] = sum_{s kept} dx_perm[row(t,s)] + dx_s[t] + dl[t] W_r."""
    d = dx_perm.shape[1]
    dx = np.zeros((T, d)) if dx_s is None else np.array(dx_s, dtype=np.float64, copy=True)
    row = np.asarray(row_of_slot).reshape(T, k)
    for s_ in range(k):
        m = row[:, s_] >= 0
        dx[m] += dx_perm[row[m, s_]]
    if dl is not None and W_r is not None:
        dx += dl @ W_r
    return dx


# --------------------------------------------------------------------------
# whole layer
# --------------------------------------------------------------------------
F64_KEYS = ("x", "W_r", "W_g", "W_u", "W_d", "Ws_g", "Ws_u", "Ws_d", "dY")


def inputs_to_f64(inp: dict) -> dict:
    """bf16-bit inputs (numpy uint16) -> float64 arrays; float32 entries
    (bias, logits_in) are kept as they are."""
    out = {}
    for key, v in inp.items():
        if v is None:
            continue
        out[key] = bf16_to_f64(v) if key in F64_KEYS else v
    return out


def layer_forward(inp: dict, k: int, capacity: int = 0, logits=None, exact_router: bool = False,
                  expert_fn=None, gates=None):
    """Forward pass of the layer.

    inp: float64 arrays x [T,d], W_g/W_u [E,H,d], W_d [E,d,H], optional shared
    Ws_g/Ws_u [Hs,d], Ws_d [d,Hs]; routing from `logits` (fp32 [T,E]) if
    given, else inp['logits_in'], else the router W_r [E,d] (+ bias [E] f32).
    exact_router: keep the router logits in float64 (finite-difference checks
    only).  expert_fn(e, x_rows) -> o_rows replaces the SwiGLU experts (pins
    only).  gates [T,k] overrides the computed gates (finite differences with
    respect to the gate values).  Returns a dict of float64 results and all
    intermediates, unrounded."""
    x = inp["x"]
    T, d = x.shape
    if logits is None:
        if inp.get("logits_in") is not None:
            logits = np.asarray(inp["logits_in"], dtype=np.float32)
        elif exact_router:
            logits = x @ inp["W_r"].T
            if inp.get("bias") is not None:
                logits = logits + np.asarray(inp["bias"], dtype=np.float64)[None, :]
        else:
            logits = router_logits(x, inp["W_r"], inp.get("bias"))
    E = logits.shape[1]
    idx, g = route_topk(logits, k)
    if gates is not None:
        g = np.asarray(gates, dtype=np.float64)
    p = permute(idx, E, capacity)
    R = int(p["offsets"][E])
    tok_of_row = p["slot_of_row"] // k
    x_perm = x[tok_of_row]
    o = np.zeros((R, d))
    out = {"logits": logits, "idx": idx, "gates": g, **p, "x_perm": x_perm}
    if expert_fn is None:
        H = inp["W_g"].shape[1]
        a = np.zeros((R, H)); u = np.zeros((R, H)); h = np.zeros((R, H))
    for e in range(E):
        r0, r1 = int(p["offsets"][e]), int(p["offsets"][e + 1])
        if r1 == r0:
            continue
        if expert_fn is None:
            a[r0:r1], u[r0:r1], h[r0:r1], o[r0:r1] = swiglu_fwd(
                x_perm[r0:r1], inp["W_g"][e], inp["W_u"][e], inp["W_d"][e])
        else:
            o[r0:r1] = expert_fn(e, x_perm[r0:r1])
    if expert_fn is None:
        out.update({"a": a, "u": u, "h": h})
    out["o"] = o
    s = None
    if inp.get("Ws_g") is not None:
        a_s, u_s, h_s, s = swiglu_fwd(x, inp["Ws_g"], inp["Ws_u"], inp["Ws_d"])
        out.update({"a_s": a_s, "u_s": u_s, "h_s": h_s, "s": s})
    out["y"] = combine(o, s, g, p["row_of_slot"], T, k)
    return out


def layer_backward(inp: dict, fwd: dict, dY=None):
    """Backward pass given the forward dict of `layer_forward` and the
    float64 upstream gradient dY [T,d] (default inp['dY']).  Returns float64
    gradients: dO, dgates, dx_perm, dW_g/dW_u/dW_d, (dx_s, dWs_*), dlogits,
    (dW_r), dx."""
    dY = inp["dY"] if dY is None else dY
    x = inp["x"]
    T, d = x.shape
    idx, gates = fwd["idx"], fwd["gates"]
    k = idx.shape[1]
    E = fwd["logits"].shape[1]
    R = int(fwd["offsets"][E])
    dO, dg = combine_bwd(dY, fwd["o"], gates, fwd["row_of_slot"], T, k)
    # experts
    H = inp["W_g"].shape[1]
    dx_perm = np.zeros((R, d))
    dWg = np.zeros((E, H, d)); dWu = np.zeros((E, H, d)); dWd = np.zeros((E, d, H))
    for e in range(E):
        r0, r1 = int(fwd["offsets"][e]), int(fwd["offsets"][e + 1])
        if r1 == r0:
            continue
        dx_e, dWg[e], dWu[e], dWd[e], _, _ = swiglu_bwd(
            fwd["x_perm"][r0:r1], inp["W_g"][e], inp["W_u"][e], inp["W_d"][e],
            fwd["a"][r0:r1], fwd["u"][r0:r1], fwd["h"][r0:r1], dO[r0:r1])
        dx_perm[r0:r1] = dx_e
    out = {"dO": dO, "dgates": dg, "dx_perm": dx_perm, "dW_g": dWg, "dW_u": dWu, "dW_d": dWd}
    dx_s = None
    if inp.get("Ws_g") is not None:
        dx_s, dWsg, dWsu, dWsd, _, _ = swiglu_bwd(
            x, inp["Ws_g"], inp["Ws_u"], inp["Ws_d"], fwd["a_s"], fwd["u_s"], fwd["h_s"], dY)
        out.update({"dx_s": dx_s, "dWs_g": dWsg, "dWs_u": dWsu, "dWs_d": dWsd})
    # router: softmax-over-S Jacobian; dropped slots have dg = 0 but stay in S
    dl = topk_bwd(gates, idx, dg, E)
    out["dlogits"] = dl
    learned = inp.get("W_r") is not None and inp.get("logits_in") is None
    if learned:
        out["dW_r"] = dl.T @ x
    out["dx"] = permute_bwd(dx_perm, dx_s, fwd["row_of_slot"], T, k,
                            dl if learned else None, inp["W_r"] if learned else None)
    return out


# --------------------------------------------------------------------------
# router balance loss (auxiliary load-balancing loss)
# --------------------------------------------------------------------------
# The pages name load-balancing-loss runs with loss weights 0.02 ... 0.5
# ("Olmo-core DDP MoE examples", "Other experiments in the report") and give
# no formula.  Reading taken: the usual auxiliary loss of top-k routing,
#   L = alpha * E * sum_e f_e P_e,
#   f_e = #{(t, s): idx[t,s] = e} / (T k)   (router assignments, before any
#                                            capacity drop),
#   P_e = (1/T) sum_t softmax(l[t, :])_e    (full softmax over the E experts
#                                            of the logits used for routing).
# f is piecewise constant in the logits, so the gradient flows through P:
#   dL/dl[t,j] = alpha E / T * p[t,j] * (f_j - sum_e f_e p[t,e]).
def router_probs(logits: np.ndarray) -> np.ndarray:
    """Full softmax over the E experts of every token (a -inf logit gives 0)."""
    l = np.asarray(logits, dtype=np.float64)
    m = l.max(axis=1, keepdims=True)
    e = np.exp(l - m)
    return e / e.sum(axis=1, keepdims=True)


def balance_loss(logits: np.ndarray, idx: np.ndarray, E: int, alpha: float):
    """Returns (L, f, P, dl): the loss, the assignment fractions, the mean
    router probabilities and dL/dlogits with f held fixed."""
    idx = np.asarray(idx)
    T, k = idx.shape
    f = np.bincount(idx.ravel().astype(np.int64), minlength=E)[:E] / float(T * k)
    p = router_probs(logits)
    P = p.mean(axis=0)
    L = alpha * E * float(f @ P)
    dl = (alpha * E / T) * p * (f[None, :] - (p @ f)[:, None])
    return L, f, P, dl
