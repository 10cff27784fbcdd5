"""A whole MoE layer call (forward and backward) through the C ABI.

`MoELayer` owns the device buffers of one shape (all allocated once with
torch; the library itself never allocates) and issues the eight C-ABI calls in
order on one stream.  It contains no arithmetic of its own: every step runs in
the CUDA library."""
from __future__ import annotations

import torch

from . import _binding as B

BF16 = torch.bfloat16


class MoELayer:
    """Buffers + call sequence for one layer shape.

    T tokens, d model width, E experts, k experts per token, H routed hidden
    width, Hs shared hidden width (0 = none), capacity (<= 0: dropless)."""

    def __init__(self, T, d, E, k, H, Hs, capacity=0, device="cuda", backward=True, balance_alpha=0.0,
                 recompute=False, fused=False):
        self.T, self.d, self.E, self.k, self.H, self.Hs, self.capacity = T, d, E, k, H, Hs, capacity
        self.balance_alpha = float(balance_alpha)
        # recompute: the forward saves no fp32 a|u; the backward rebuilds them
        # (moe_grouped_swiglu_recompute) into au / au_s, which then only have
        # to live through the backward call (scratch that layers can share)
        self.recompute = bool(recompute)
        # fused: the permutation is fused into the GEMMs' operand loads (row
        # gathers from x and dY) and the combine into the shared expert's
        # down-projection epilogue: no x_perm, dY_perm or s; o_perm holds the
        # expert outputs by slot (moe_grouped_swiglu_fused)
        self.fused = bool(fused)
        dev = torch.device(device)
        R = T * k
        e = lambda *shape, dt=BF16: torch.empty(*shape, dtype=dt, device=dev)  # noqa: E731
        self.logits = e(T, E, dt=torch.float32)
        self.idx = e(T, k, dt=torch.int32)
        self.gates = e(T, k, dt=torch.float32)
        self.counts_raw = e(E, dt=torch.int32)
        self.counts = e(E, dt=torch.int32)
        self.offsets = e(E + 1, dt=torch.int32)
        self.row_of_slot = e(R, dt=torch.int32)
        self.slot_of_row = e(R, dt=torch.int32)
        self.x_perm = None if self.fused else e(R, d)
        self.au = e(R, 2 * H, dt=torch.float32) if backward else None
        self.h = e(R, H)
        # the terms of the per-token sums (expert outputs, shared output,
        # input-gradient rows) in fp16
        self.o_perm = e(R, d, dt=torch.float16)
        self.au_s = e(T, 2 * Hs, dt=torch.float32) if (Hs and backward) else None
        self.h_s = e(T, Hs) if Hs else None
        self.s = e(T, d, dt=torch.float16) if (Hs and not self.fused) else None
        self.y = e(T, d)
        if self.balance_alpha > 0:
            # auxiliary load-balancing loss (device scalar), mean router
            # probabilities and the loss gradient of the logits
            self.lbl_loss = e(1, dt=torch.float32)
            self.lbl_P = e(E, dt=torch.float32)
            self.dlogits_lbl = e(T, E, dt=torch.float32) if backward else None
        self.ws_bytes = B.moe_workspace_size(T, d, E, k, H, Hs)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        if backward:
            self.dY_perm = None if self.fused else e(R, d)
            self.dgates = e(T, k, dt=torch.float32)
            self.dx_perm = e(R, d, dt=torch.float16)
            self.dx_s = e(T, d, dt=torch.float16) if Hs else None
            self.dW_g = e(E, H, d)
            self.dW_u = e(E, H, d)
            self.dW_d = e(E, d, H)
            self.dWs_g = e(Hs, d) if Hs else None
            self.dWs_u = e(Hs, d) if Hs else None
            self.dWs_d = e(d, Hs) if Hs else None
            self.dlogits = e(T, E, dt=torch.float32)
            # scale word of the fp16 input-gradient terms (the max |dY| pattern)
            self.dx_scale = e(1, dt=torch.int32)
            self.dW_r = e(E, d, dt=torch.float32)
            self.dx = e(T, d)

    # ------------------------------------------------------------------
    def forward(self, x, p, logits_in=None, stream=None):
        """x [T,d] bf16; p: dict of device weights (W_r, bias, W_g, W_u, W_d,
        Ws_g, Ws_u, Ws_d).  Returns y [T,d] bf16 (self.y)."""
        T, d, E, k, H, Hs = self.T, self.d, self.E, self.k, self.H, self.Hs
        B.moe_route_topk(x, p.get("W_r"), p.get("bias"), logits_in, T, d, E, k,
                         None if logits_in is not None else self.logits, self.idx, self.gates,
                         self.ws, self.ws_bytes, stream)
        B.moe_permute(None if self.fused else x, self.idx, T, d, E, k, self.capacity, self.counts_raw, self.counts,
                      self.offsets, self.row_of_slot, self.slot_of_row, self.x_perm, self.ws, self.ws_bytes, stream)
        if self.balance_alpha > 0:
            B.moe_router_balance_loss(logits_in if logits_in is not None else self.logits, self.counts_raw, T, E, k,
                                      self.balance_alpha, self.lbl_loss, self.lbl_P, self.dlogits_lbl, self.ws,
                                      self.ws_bytes, stream)
        save = not self.recompute
        if self.fused:
            B.moe_grouped_swiglu_fused(x, self.slot_of_row, self.row_of_slot, self.gates, self.offsets, T, d, E, k, H,
                                       Hs, p["W_g"], p["W_u"], p["W_d"], p.get("Ws_g"), p.get("Ws_u"), p.get("Ws_d"),
                                       self.au if save else None, self.h, self.o_perm,
                                       self.au_s if save else None, self.h_s, self.y, stream)
            return self.y
        B.moe_grouped_swiglu(self.x_perm, self.offsets, x, T, d, E, k, H, Hs, p["W_g"], p["W_u"], p["W_d"],
                             p.get("Ws_g"), p.get("Ws_u"), p.get("Ws_d"), self.au if save else None, self.h,
                             self.o_perm, self.au_s if save else None, self.h_s, self.s, self.ws, self.ws_bytes,
                             stream)
        B.moe_unpermute_combine(self.o_perm, self.s, self.gates, self.row_of_slot, T, d, k, self.y, stream)
        return self.y

    def backward(self, x, dY, p, learned_router=True, stream=None):
        """Backward of the last forward for upstream dY [T,d] bf16.  Fills
        dx, dW_g/u/d, dWs_*, dgates, dlogits and (learned router) dW_r; with
        balance_alpha > 0 the load-balancing loss's gradient is included in
        dlogits, dW_r and dx."""
        T, d, E, k, H, Hs = self.T, self.d, self.E, self.k, self.H, self.Hs
        if self.recompute and self.fused:
            B.moe_grouped_swiglu_recompute_fused(x, self.slot_of_row, self.offsets, T, d, E, k, H, Hs, p["W_g"],
                                                 p["W_u"], p.get("Ws_g"), p.get("Ws_u"), self.au, self.au_s, stream)
        elif self.recompute:
            B.moe_grouped_swiglu_recompute(self.x_perm, self.offsets, x, T, d, E, k, H, Hs, p["W_g"], p["W_u"],
                                           p.get("Ws_g"), p.get("Ws_u"), self.au, self.au_s, stream)
        if not self.fused:
            B.moe_unpermute_combine_bwd(dY, self.row_of_slot, T, d, k, self.dY_perm, stream)
        B.moe_grouped_swiglu_bwd(self.dY_perm, dY, self.gates, self.row_of_slot, self.slot_of_row, self.offsets,
                                 self.x_perm, x, self.au, self.au_s, T, d, E, k, H, Hs, p["W_g"], p["W_u"],
                                 p["W_d"], p.get("Ws_g"), p.get("Ws_u"), p.get("Ws_d"), self.dx_perm, self.dx_s,
                                 self.dW_g, self.dW_u, self.dW_d, self.dWs_g, self.dWs_u, self.dWs_d, self.dgates,
                                 self.ws, self.ws_bytes, stream, dx_scale=self.dx_scale)
        lr = learned_router and p.get("W_r") is not None
        B.moe_route_topk_bwd(self.dgates, self.gates, self.idx, x if lr else None, T, d, E, k, self.dlogits,
                             self.dW_r if lr else None, self.ws, self.ws_bytes, stream,
                             dlogits_add=self.dlogits_lbl if self.balance_alpha > 0 else None)
        B.moe_permute_bwd(self.dx_perm, self.dx_s, self.row_of_slot, self.dlogits if lr else None,
                          p.get("W_r") if lr else None, T, d, E, k, self.dx, self.ws, self.ws_bytes, stream,
                          dx_scale=self.dx_scale)
        return self.dx
