"""The C++ oracle of the MoE layer (oracle/moe_oracle.cpp), with the same
Python interface as the numpy oracle (oracle/moe_oracle.py): layer_forward,
layer_backward, router_logits, route_topk, permute, bf16_to_f64,
inputs_to_f64, capacity_of.

TEST INFRASTRUCTURE ONLY.  Only the tests, `__graft_entry__.smoke()` and the
bench's CPU-baseline / reference leg may import this module; the CUDA
library never loads it and the two share no code.

The library is built on first import (oracle/build_oracle.py, the host C++
compiler).  All arithmetic happens in the C++ code; this module only
allocates the result arrays and passes pointers."""
from __future__ import annotations

import ctypes

import numpy as np

from . import build_oracle

_lib = ctypes.CDLL(build_oracle.build())
_P = ctypes.c_void_p
_I = ctypes.c_int
_LL = ctypes.c_longlong

_lib.orc_set_threads.argtypes = [_I]
_lib.orc_threads.restype = _I
_lib.orc_bf16_to_f64.argtypes = [_P, _LL, _P]
_lib.orc_router_logits.argtypes = [_P, _P, _P, _I, _I, _I, _P]
_lib.orc_route_topk.argtypes = [_P, _I, _I, _I, _P, _P]
_lib.orc_permute.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]
_lib.orc_permute.restype = _LL
_lib.orc_layer_forward.argtypes = [_I] * 7 + [_P] * 4 + [_I, _P, _I] + [_P] * 6 + [_P] * 19
_lib.orc_layer_forward.restype = _LL
_lib.orc_layer_backward.argtypes = [_I] * 6 + [_P, _P, _I] + [_P] * 6 + [_P] * 13 + [_P] * 13


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def set_threads(n: int) -> None:
    """Worker threads of the oracle (0: one per host core)."""
    _lib.orc_set_threads(int(n))


def threads() -> int:
    return int(_lib.orc_threads())


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _lib.orc_bf16_to_f64(_p(b), b.size, _p(out))
    return out


F64_KEYS = ("x", "W_r", "W_g", "W_u", "W_d", "Ws_g", "Ws_u", "Ws_d", "dY")


def inputs_to_f64(inp: dict) -> dict:
    """bf16-bit inputs (uint16) -> float64 arrays; float32 entries (bias,
    logits_in) are kept as they are."""
    return {k: (bf16_to_f64(v) if k in F64_KEYS else v) for k, v in inp.items() if v is not None}


def capacity_of(T: int, k: int, E: int, factor_num: int = 5, factor_den: int = 4) -> int:
    """C = ceil(factor * T * k / E) in integers (factor = num/den)."""
    return (factor_num * T * k + factor_den * E - 1) // (factor_den * E)


def router_logits(x, W_r, bias=None) -> np.ndarray:
    x, W_r = _f64(x), _f64(W_r)
    T, d = x.shape
    E = W_r.shape[0]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = np.empty((T, E), dtype=np.float32)
    _lib.orc_router_logits(_p(x), _p(W_r), _p(b), T, d, E, _p(out))
    return out


def route_topk(logits, k: int):
    l = np.asarray(logits)
    l = np.ascontiguousarray(l.astype(np.float32).astype(np.float64) if l.dtype != np.float64 else l)
    T, E = l.shape
    idx = np.empty((T, k), dtype=np.int32)
    gates = np.empty((T, k), dtype=np.float64)
    _lib.orc_route_topk(_p(l), T, E, k, _p(idx), _p(gates))
    return idx, gates


def permute(idx, E: int, capacity: int = 0):
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    cr, c = np.empty(E, dtype=np.int64), np.empty(E, dtype=np.int64)
    off = np.empty(E + 1, dtype=np.int64)
    rank = np.empty(T * k, dtype=np.int64)
    row = np.empty(T * k, dtype=np.int64)
    sor = np.full(T * k, -1, dtype=np.int64)
    R = _lib.orc_permute(_p(idx), T, E, k, capacity, _p(cr), _p(c), _p(off), _p(rank), _p(row), _p(sor))
    return {"counts_raw": cr, "counts": c, "offsets": off, "rank": rank.reshape(T, k),
            "kept": (row >= 0).reshape(T, k), "row_of_slot": row, "slot_of_row": sor[:R]}


def _is_identity(expert_fn) -> bool:
    probe = np.arange(12, dtype=np.float64).reshape(3, 4) - 5.5
    return np.array_equal(expert_fn(0, probe.copy()), probe)


def layer_forward(inp: dict, k: int, capacity: int = 0, logits=None, exact_router: bool = False,
                  expert_fn=None, gates=None):
    """Forward pass; the same arguments and result keys as the numpy oracle's
    layer_forward (expert_fn: only the identity o = x is supported)."""
    identity = False
    if expert_fn is not None:
        if not _is_identity(expert_fn):
            raise NotImplementedError("the C++ oracle supports identity experts only")
        identity = True
    x = _f64(inp["x"])
    T, d = x.shape
    W_g = _f64(inp["W_g"]) if not identity else None
    E = inp["W_r"].shape[0] if inp.get("W_r") is not None else None
    logits_in = None
    if logits is not None:
        logits_in = np.asarray(logits)
    elif inp.get("logits_in") is not None:
        logits_in = np.asarray(inp["logits_in"], dtype=np.float32)
    if logits_in is not None:
        E = logits_in.shape[1]
        given_dtype = logits_in.dtype
        logits_in = np.ascontiguousarray(logits_in.astype(np.float64))
    H = inp["W_g"].shape[1] if inp.get("W_g") is not None else 0
    Hs = inp["Ws_g"].shape[0] if inp.get("Ws_g") is not None and not identity else 0
    R = T * k
    W_r = _f64(inp.get("W_r"))
    bias = None if inp.get("bias") is None else np.ascontiguousarray(inp["bias"], dtype=np.float32)
    g_in = _f64(gates)
    out = {
        "logits": np.empty((T, E)), "idx": np.empty((T, k), dtype=np.int32), "gates": np.empty((T, k)),
        "counts_raw": np.empty(E, dtype=np.int64), "counts": np.empty(E, dtype=np.int64),
        "offsets": np.empty(E + 1, dtype=np.int64), "rank": np.empty((T, k), dtype=np.int64),
        "row_of_slot": np.empty(T * k, dtype=np.int64), "slot_of_row": np.full(R, -1, dtype=np.int64),
        "x_perm": np.empty((R, d)), "a": np.zeros((R, H)), "u": np.zeros((R, H)), "h": np.zeros((R, H)),
        "o": np.zeros((R, d)), "y": np.empty((T, d)),
    }
    sh = {"a_s": np.empty((T, Hs)), "u_s": np.empty((T, Hs)), "h_s": np.empty((T, Hs)), "s": np.empty((T, d))} \
        if Hs else {"a_s": None, "u_s": None, "h_s": None, "s": None}
    ws = [_f64(inp.get(n)) if not identity else None for n in ("W_g", "W_u", "W_d")]
    wss = [_f64(inp.get(n)) if Hs else None for n in ("Ws_g", "Ws_u", "Ws_d")]
    R = _lib.orc_layer_forward(
        T, d, E, k, H, Hs, capacity, _p(x), _p(W_r), _p(bias), _p(logits_in), int(bool(exact_router)), _p(g_in),
        int(identity), *[_p(v) for v in ws], *[_p(v) for v in wss],
        _p(out["logits"]), _p(out["idx"]), _p(out["gates"]), _p(out["counts_raw"]), _p(out["counts"]),
        _p(out["offsets"]), _p(out["rank"]), _p(out["row_of_slot"]), _p(out["slot_of_row"]), _p(out["x_perm"]),
        _p(out["a"]), _p(out["u"]), _p(out["h"]), _p(out["o"]),
        _p(sh["a_s"]), _p(sh["u_s"]), _p(sh["h_s"]), _p(sh["s"]), _p(out["y"]))
    for key in ("slot_of_row", "x_perm", "a", "u", "h", "o"):
        out[key] = out[key][:R]
    out["kept"] = (out["row_of_slot"] >= 0).reshape(T, k)
    if logits_in is not None:
        out["logits"] = out["logits"].astype(given_dtype) if given_dtype != np.float64 else out["logits"]
    elif not exact_router:
        out["logits"] = out["logits"].astype(np.float32)
    if identity:
        for key in ("a", "u", "h"):
            del out[key]
    if Hs:
        out.update(sh)
    out["_inp_shapes"] = (T, d, E, k, H, Hs)
    return out


def layer_backward(inp: dict, fwd: dict, dY=None):
    """Backward pass; the same arguments and result keys as the numpy
    oracle's layer_backward."""
    T, d, E, k, H, Hs = fwd["_inp_shapes"]
    dY = _f64(inp["dY"] if dY is None else dY)
    x = _f64(inp["x"])
    learned = inp.get("W_r") is not None and inp.get("logits_in") is None
    W_r = _f64(inp["W_r"]) if learned else None
    R = int(fwd["offsets"][E])
    ws = [_f64(inp[n]) for n in ("W_g", "W_u", "W_d")]
    wss = [_f64(inp[n]) if Hs else None for n in ("Ws_g", "Ws_u", "Ws_d")]
    out = {"dO": np.zeros((max(R, 1), d)), "dgates": np.empty((T, k)), "dx_perm": np.zeros((max(R, 1), d)),
           "dW_g": np.empty((E, H, d)), "dW_u": np.empty((E, H, d)), "dW_d": np.empty((E, d, H)),
           "dlogits": np.empty((T, E)), "dx": np.empty((T, d))}
    sh = {"dx_s": np.empty((T, d)), "dWs_g": np.empty((Hs, d)), "dWs_u": np.empty((Hs, d)),
          "dWs_d": np.empty((d, Hs))} if Hs else {"dx_s": None, "dWs_g": None, "dWs_u": None, "dWs_d": None}
    dW_r = np.empty((E, d)) if learned else None
    f = {key: _f64(fwd[key]) for key in ("gates", "x_perm", "a", "u", "h", "o")}
    fs = {key: (_f64(fwd[key]) if Hs else None) for key in ("a_s", "u_s", "h_s")}
    idx = np.ascontiguousarray(fwd["idx"], dtype=np.int32)
    off = np.ascontiguousarray(fwd["offsets"], dtype=np.int64)
    row = np.ascontiguousarray(fwd["row_of_slot"], dtype=np.int64)
    _lib.orc_layer_backward(
        T, d, E, k, H, Hs, _p(x), _p(W_r), int(learned), *[_p(v) for v in ws], *[_p(v) for v in wss], _p(dY),
        _p(idx), _p(f["gates"]), _p(off), _p(row), _p(f["x_perm"]), _p(f["a"]), _p(f["u"]), _p(f["h"]),
        _p(f["o"]), _p(fs["a_s"]), _p(fs["u_s"]), _p(fs["h_s"]),
        _p(out["dO"]), _p(out["dgates"]), _p(out["dx_perm"]), _p(out["dW_g"]), _p(out["dW_u"]), _p(out["dW_d"]),
        _p(sh["dx_s"]), _p(sh["dWs_g"]), _p(sh["dWs_u"]), _p(sh["dWs_d"]), _p(out["dlogits"]), _p(dW_r),
        _p(out["dx"]))
    out["dO"] = out["dO"][:R]
    out["dx_perm"] = out["dx_perm"][:R]
    if Hs:
        out.update(sh)
    if learned:
        out["dW_r"] = dW_r
    return out
