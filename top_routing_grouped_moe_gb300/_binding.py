"""ctypes binding of the C ABI (include/moe.h): the same function names,
argument marshalling only.  Tensors are passed as device pointers
(torch.Tensor.data_ptr()); every step runs in the CUDA library.

Importing this module loads lib/libmoe_gb300.so; if the library has not been
built, the import fails loudly (there is no fallback path)."""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE_BOUNDS = 6
MOE_ERR_RANGE = 7


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: status {status} ({msg})")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"CUDA library not built: {LIB_PATH} is missing "
                          "(run `python -m top_routing_grouped_moe_gb300.build`)")
    return ctypes.CDLL(LIB_PATH)


_lib = _load()

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t

# name -> argument kinds ('p' pointer/tensor, 'i' int, 'f' float, 'z' size_t, 's' stream)
SIGNATURES = {
    "moe_route_topk": "pppp" + "iiii" + "ppp" + "pz" + "s",
    "moe_permute": "pp" + "iiiii" + "pppppp" + "pz" + "s",
    "moe_permute_static": "pp" + "iiiii" + "pppppp" + "s",
    "moe_grouped_swiglu": "ppp" + "iiiiii" + "pppppp" + "pppppp" + "pz" + "s",
    "moe_grouped_swiglu_recompute": "ppp" + "iiiiii" + "pppp" + "pp" + "s",
    "moe_grouped_swiglu_fused": "ppppp" + "iiiiii" + "pppppp" + "ppp" + "ppp" + "s",
    "moe_grouped_swiglu_recompute_fused": "ppp" + "iiiiii" + "pppp" + "pp" + "s",
    "moe_unpermute_combine": "pppp" + "iii" + "p" + "s",
    "moe_unpermute_combine_bwd": "pp" + "iii" + "p" + "s",
    "moe_grouped_swiglu_bwd": "pppppppppp" + "iiiiii" + "pppppp" + "pp" + "pppppp" + "pp" + "pz" + "s",
    "moe_route_topk_bwd": "pppp" + "iiii" + "ppp" + "pz" + "s",
    "moe_router_balance_loss": "pp" + "iii" + "f" + "ppp" + "pz" + "s",
    "moe_permute_bwd": "ppppp" + "iiii" + "pp" + "pz" + "s",
    "moe_mxfp8_quantize": "p" + "Li" + "pp" + "s",
    "moe_mxfp8_quantize_gate_up": "pp" + "iii" + "pp" + "s",
    "moe_permute_mxfp8": "pp" + "iiiii" + "pppppp" + "pp" + "pz" + "s",
    "moe_grouped_swiglu_mxfp8": "pppppp" + "iiiiii" + "pppppppp" + "pppp" + "pp" + "s",
    "moe_unpermute_combine_mxfp8": "pppp" + "iiii" + "p" + "s",
    "moe_selftest_group_maps": "",
    "moe_selftest_wait_timeout": "i" + "s",
}

_CT = {"p": _P, "i": _I, "L": ctypes.c_longlong, "f": ctypes.c_float, "z": _SZ, "s": _P}

for _name, _sig in SIGNATURES.items():
    _f = getattr(_lib, _name)
    _f.argtypes = [_CT[c] for c in _sig]
    _f.restype = _I

_lib.moe_version.restype = _I
_lib.moe_version.argtypes = []
_lib.moe_status_string.restype = ctypes.c_char_p
_lib.moe_status_string.argtypes = [_I]
_lib.moe_last_cuda_error.restype = _I
_lib.moe_last_cuda_error.argtypes = []
_lib.moe_device_status.restype = _I
_lib.moe_device_status.argtypes = [ctypes.POINTER(_I)]
_lib.moe_workspace_size.restype = _I
_lib.moe_workspace_size.argtypes = [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_SZ)]
_lib.moe_mxfp8_rows.restype = _I
_lib.moe_mxfp8_rows.argtypes = [_I, _I, _I, ctypes.POINTER(ctypes.c_longlong)]
_lib.moe_mxfp8_scales_bytes.restype = _I
_lib.moe_mxfp8_scales_bytes.argtypes = [ctypes.c_longlong, _I, ctypes.POINTER(_SZ)]
_lib.moe_timing_begin.restype = _I
_lib.moe_timing_begin.argtypes = [ctypes.POINTER(_P), _I]
_lib.moe_timing_end.restype = _I
_lib.moe_timing_end.argtypes = [ctypes.POINTER(_I)]
_lib.moe_timing_name.restype = ctypes.c_char_p
_lib.moe_timing_name.argtypes = [_I]
_lib.moe_timing_record.restype = _I
_lib.moe_timing_record.argtypes = [_P, _P]


def _ptr(v):
    if v is None:
        return None
    if isinstance(v, torch.Tensor):
        return ctypes.c_void_p(v.data_ptr())
    return ctypes.c_void_p(int(v))


def _stream(v):
    if v is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(v, torch.cuda.Stream):
        return ctypes.c_void_p(v.cuda_stream)
    return ctypes.c_void_p(int(v))


def status_string(status: int) -> str:
    return _lib.moe_status_string(int(status)).decode()


def _call(name: str, *args):
    sig = SIGNATURES[name]
    if len(args) != len(sig):
        raise TypeError(f"{name} takes {len(sig)} arguments ({len(args)} given)")
    conv = []
    for kind, a in zip(sig, args):
        if kind == "p":
            conv.append(_ptr(a))
        elif kind == "s":
            conv.append(_stream(a))
        elif kind == "f":
            conv.append(float(a))
        else:
            conv.append(int(a))
    rc = getattr(_lib, name)(*conv)
    if rc != MOE_OK:
        msg = status_string(rc)
        if rc == MOE_ERR_CUDA:
            msg += f", cudaError {_lib.moe_last_cuda_error()}"
        raise MoEError(name, rc, msg)
    return rc


def moe_version() -> int:
    return _lib.moe_version()


def moe_device_status() -> int:
    v = _I(0)
    rc = _lib.moe_device_status(ctypes.byref(v))
    if rc != MOE_OK:
        raise MoEError("moe_device_status", rc, status_string(rc))
    return v.value


def moe_workspace_size(T, d, E, k, H, Hs) -> int:
    b = _SZ(0)
    rc = _lib.moe_workspace_size(T, d, E, k, H, Hs, ctypes.byref(b))
    if rc != MOE_OK:
        raise MoEError("moe_workspace_size", rc, status_string(rc))
    return b.value


class LaunchTimer:
    """Times every kernel launch of the library's calls made inside a `with`
    block in this thread (moe_timing_begin / moe_timing_end), with CUDA
    events recorded on each launch's own stream.  After the block and a
    synchronize, `launches()` gives [(kernel name, ms)].  Inside stream
    capture the records become event-record nodes of the graph: after each
    replay and a synchronize, `launches()` gives that replay's times."""

    def __init__(self, capacity=256, stream=None):
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(capacity + 1)]
        self.stream = stream
        # torch creates the CUDA event at its first record: record each once so
        # that every handle exists before the library records it
        for e in self.events:
            e.record(stream if stream is not None else torch.cuda.current_stream())
        self._arr = (_P * capacity)(*[ctypes.c_void_p(e.cuda_event) for e in self.events[:capacity]])
        self.n = 0
        self.names = []

    def __enter__(self):
        rc = _lib.moe_timing_begin(self._arr, len(self._arr))
        if rc != MOE_OK:
            raise MoEError("moe_timing_begin", rc, status_string(rc))
        return self

    def __exit__(self, *exc):
        n = _I(0)
        rc = _lib.moe_timing_end(ctypes.byref(n))
        if rc != MOE_OK:
            raise MoEError("moe_timing_end", rc, status_string(rc))
        self.n = n.value
        if self.n > len(self._arr):
            raise RuntimeError(f"LaunchTimer: {self.n} launches, capacity {len(self._arr)}")
        self.names = [_lib.moe_timing_name(i).decode() for i in range(self.n)]
        # the end of the last launch (a graph node too, when capturing)
        s = self.stream if self.stream is not None else torch.cuda.current_stream()
        rc = _lib.moe_timing_record(ctypes.c_void_p(self.events[self.n].cuda_event), ctypes.c_void_p(s.cuda_stream))
        if rc != MOE_OK:
            raise MoEError("moe_timing_record", rc, status_string(rc))
        return False

    def launches(self):
        return [(self.names[i], self.events[i].elapsed_time(self.events[i + 1])) for i in range(self.n)]


def moe_route_topk(x, W_r, bias, logits_in, T, d, E, k, logits, topk_idx, gates, ws, ws_bytes, stream=None):
    return _call("moe_route_topk", x, W_r, bias, logits_in, T, d, E, k, logits, topk_idx, gates, ws, ws_bytes,
                 stream)


def moe_permute(x, topk_idx, T, d, E, k, capacity, counts_raw, counts, offsets, row_of_slot, slot_of_row, x_perm,
                ws, ws_bytes, stream=None):
    return _call("moe_permute", x, topk_idx, T, d, E, k, capacity, counts_raw, counts, offsets, row_of_slot,
                 slot_of_row, x_perm, ws, ws_bytes, stream)


def moe_permute_static(x, topk_idx, T, d, E, k, capacity, counts_raw, counts, offsets, row_of_slot, slot_of_row,
                       x_perm, stream=None):
    return _call("moe_permute_static", x, topk_idx, T, d, E, k, capacity, counts_raw, counts, offsets,
                 row_of_slot, slot_of_row, x_perm, stream)


def moe_grouped_swiglu(x_perm, offsets, x, T, d, E, k, H, Hs, W_g, W_u, W_d, Ws_g, Ws_u, Ws_d, au, h, o_perm,
                       au_s, h_s, s, ws, ws_bytes, stream=None):
    return _call("moe_grouped_swiglu", x_perm, offsets, x, T, d, E, k, H, Hs, W_g, W_u, W_d, Ws_g, Ws_u, Ws_d, au,
                 h, o_perm, au_s, h_s, s, ws, ws_bytes, stream)


def moe_grouped_swiglu_recompute(x_perm, offsets, x, T, d, E, k, H, Hs, W_g, W_u, Ws_g, Ws_u, au, au_s,
                                 stream=None):
    return _call("moe_grouped_swiglu_recompute", x_perm, offsets, x, T, d, E, k, H, Hs, W_g, W_u, Ws_g, Ws_u, au,
                 au_s, stream)


def moe_grouped_swiglu_fused(x, slot_of_row, row_of_slot, gates, offsets, T, d, E, k, H, Hs, W_g, W_u, W_d, Ws_g,
                             Ws_u, Ws_d, au, h, o_slot, au_s, h_s, y, stream=None):
    return _call("moe_grouped_swiglu_fused", x, slot_of_row, row_of_slot, gates, offsets, T, d, E, k, H, Hs, W_g,
                 W_u, W_d, Ws_g, Ws_u, Ws_d, au, h, o_slot, au_s, h_s, y, stream)


def moe_grouped_swiglu_recompute_fused(x, slot_of_row, offsets, T, d, E, k, H, Hs, W_g, W_u, Ws_g, Ws_u, au, au_s,
                                       stream=None):
    return _call("moe_grouped_swiglu_recompute_fused", x, slot_of_row, offsets, T, d, E, k, H, Hs, W_g, W_u, Ws_g,
                 Ws_u, au, au_s, stream)


def moe_unpermute_combine(o_perm, s, gates, row_of_slot, T, d, k, y, stream=None):
    return _call("moe_unpermute_combine", o_perm, s, gates, row_of_slot, T, d, k, y, stream)


def moe_unpermute_combine_bwd(dY, row_of_slot, T, d, k, dY_perm, stream=None):
    return _call("moe_unpermute_combine_bwd", dY, row_of_slot, T, d, k, dY_perm, stream)


def moe_grouped_swiglu_bwd(dY_perm, dY, gates, row_of_slot, slot_of_row, offsets, x_perm, x, au, au_s, T, d, E, k,
                           H, Hs, W_g, W_u, W_d, Ws_g, Ws_u, Ws_d, dx_perm, dx_s, dW_g, dW_u, dW_d, dWs_g, dWs_u,
                           dWs_d, dgates, ws, ws_bytes, stream=None, dx_scale=None):
    """dx_scale: optional int32/uint32 [1] device word (see moe.h): the fp16
    terms dx_perm / dx_s are stored divided by 2^e of max |dY|."""
    return _call("moe_grouped_swiglu_bwd", dY_perm, dY, gates, row_of_slot, slot_of_row, offsets, x_perm, x, au,
                 au_s, T, d, E, k, H, Hs, W_g, W_u, W_d, Ws_g, Ws_u, Ws_d, dx_perm, dx_s, dW_g, dW_u, dW_d, dWs_g,
                 dWs_u, dWs_d, dgates, dx_scale, ws, ws_bytes, stream)


def moe_route_topk_bwd(dgates, gates, topk_idx, x, T, d, E, k, dlogits, dW_r, ws, ws_bytes, stream=None,
                       dlogits_add=None):
    return _call("moe_route_topk_bwd", dgates, gates, topk_idx, x, T, d, E, k, dlogits, dW_r, dlogits_add, ws,
                 ws_bytes, stream)


def moe_router_balance_loss(logits, counts_raw, T, E, k, alpha, loss, P_mean, dlogits_lbl, ws, ws_bytes, stream=None):
    return _call("moe_router_balance_loss", logits, counts_raw, T, E, k, alpha, loss, P_mean, dlogits_lbl, ws,
                 ws_bytes, stream)


def moe_permute_bwd(dx_perm, dx_s, row_of_slot, dlogits, W_r, T, d, E, k, dx, ws, ws_bytes, stream=None,
                    dx_scale=None):
    """dx_scale: the word moe_grouped_swiglu_bwd wrote for these terms (or None)."""
    return _call("moe_permute_bwd", dx_perm, dx_s, row_of_slot, dlogits, W_r, T, d, E, k, dx, dx_scale, ws,
                 ws_bytes, stream)


def moe_mxfp8_rows(T, E, k) -> int:
    v = ctypes.c_longlong(0)
    rc = _lib.moe_mxfp8_rows(T, E, k, ctypes.byref(v))
    if rc != MOE_OK:
        raise MoEError("moe_mxfp8_rows", rc, status_string(rc))
    return v.value


def moe_mxfp8_scales_bytes(rows, cols) -> int:
    v = _SZ(0)
    rc = _lib.moe_mxfp8_scales_bytes(rows, cols, ctypes.byref(v))
    if rc != MOE_OK:
        raise MoEError("moe_mxfp8_scales_bytes", rc, status_string(rc))
    return v.value


def moe_mxfp8_quantize(src, rows, cols, codes, scales, stream=None):
    return _call("moe_mxfp8_quantize", src, rows, cols, codes, scales, stream)


def moe_mxfp8_quantize_gate_up(W_g, W_u, E, H, d, codes, scales, stream=None):
    return _call("moe_mxfp8_quantize_gate_up", W_g, W_u, E, H, d, codes, scales, stream)


def moe_permute_mxfp8(x, topk_idx, T, d, E, k, capacity, counts_raw, counts, offsets, mx_offsets, row_of_slot,
                      slot_of_row, x_codes, x_scales, ws, ws_bytes, stream=None):
    return _call("moe_permute_mxfp8", x, topk_idx, T, d, E, k, capacity, counts_raw, counts, offsets, mx_offsets,
                 row_of_slot, slot_of_row, x_codes, x_scales, ws, ws_bytes, stream)


def moe_grouped_swiglu_mxfp8(x_codes, x_scales, mx_offsets, counts, xs_codes, xs_scales, T, d, E, k, H, Hs,
                             Wgu_codes, Wgu_scales, Wd_codes, Wd_scales, Wsgu_codes, Wsgu_scales, Wsd_codes,
                             Wsd_scales, h_codes, h_scales, hs_codes, hs_scales, o_perm, s, stream=None):
    return _call("moe_grouped_swiglu_mxfp8", x_codes, x_scales, mx_offsets, counts, xs_codes, xs_scales, T, d, E, k,
                 H, Hs, Wgu_codes, Wgu_scales, Wd_codes, Wd_scales, Wsgu_codes, Wsgu_scales, Wsd_codes, Wsd_scales,
                 h_codes, h_scales, hs_codes, hs_scales, o_perm, s, stream)


def moe_unpermute_combine_mxfp8(o_perm, s, gates, row_of_slot, T, d, E, k, y, stream=None):
    return _call("moe_unpermute_combine_mxfp8", o_perm, s, gates, row_of_slot, T, d, E, k, y, stream)


def moe_selftest_group_maps():
    return _call("moe_selftest_group_maps")


def moe_selftest_wait_timeout(limit_us, stream=None):
    return _call("moe_selftest_wait_timeout", limit_us, stream)
