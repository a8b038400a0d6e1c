"""A routed MoE expert-MLP layer of fixed size on one GPU: owns every buffer the
C ABI needs (allocated once with torch, reused by every call) and strings the
entry points together.

Router (optional): moe_router_topk (logits -> topk_ids, topk_w); after the backward,
moe_router_weight_grad + moe_router_backward (-> d_logits).
Forward:  moe_route_permute -> moe_expert_mlp_fwd -> moe_combine(topk_w)
Backward: moe_expert_mlp_bwd (which also reduces the routed dX to tokens; or, with
          reduce_in_backward=False, moe_expert_mlp_bwd -> moe_combine(NULL))

Buffer shapes are fixed by (T, K, E, D, I, align), so a forward/backward pair can
be captured once in a CUDA graph and replayed with new inputs and routings.
"""
from __future__ import annotations

import torch

from . import binding as B


class MoEExpertMLP:
    """`skip_padding`: pass the routing's per-expert counts to the GEMMs so that they
    compute only the real rows of each expert's last row tile (rounded up to 32); off,
    every padded row is computed.  `reduce_in_backward`: moe_expert_mlp_bwd reduces the
    routed dX to tokens itself, beside its weight-gradient GEMMs; off, a separate
    moe_combine call does it afterwards.  The results are the same bit for bit."""

    def __init__(self, T: int, K: int, E: int, D: int, I: int, align: int = 128,
                 device: str | torch.device = "cuda", skip_padding: bool = True,
                 reduce_in_backward: bool = True):
        self.T, self.K, self.E, self.D, self.I, self.align = T, K, E, D, I, align
        self.skip_padding = skip_padding
        self.reduce_in_backward = reduce_in_backward
        dev = torch.device(device)
        self.device = dev
        self.cap = B.moe_capacity(T, K, E, align)
        if self.cap == 0 and T * K > 0:
            raise ValueError("invalid layer sizes")
        cap = max(self.cap, 1)
        i32, f32, bf = torch.int32, torch.float32, torch.bfloat16
        self.counts = torch.zeros(E, dtype=i32, device=dev)
        self.offsets = torch.zeros(E + 1, dtype=i32, device=dev)
        self.perm_src = torch.empty(cap, dtype=i32, device=dev)
        self.inv_perm = torch.empty(max(T * K, 1), dtype=i32, device=dev)
        self.w_perm = torch.empty(cap, dtype=f32, device=dev)
        self.x_perm = torch.empty(cap, D, dtype=bf, device=dev)
        self.y_perm = torch.empty(cap, D, dtype=bf, device=dev)
        self.y = torch.empty(T, D, dtype=bf, device=dev)
        self.dx_perm = torch.empty(cap, D, dtype=bf, device=dev)
        self.dx = torch.empty(T, D, dtype=bf, device=dev)
        self.dw_gate = torch.empty(E, D, I, dtype=f32, device=dev)
        self.dw_up = torch.empty(E, D, I, dtype=f32, device=dev)
        self.dw_down = torch.empty(E, I, D, dtype=f32, device=dev)
        ws = B.moe_workspace_bytes(T, K, E, D, I, align)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
        B.moe_workspace_init(self.workspace)
        self._topk_w = None
        self._x = None

    def forward(self, x, topk_ids, topk_w, w_gate, w_up, w_down, stream=None, out=None):
        """Y [T, D] bf16 = sum_k topk_w[t,k] * SwiGLU-MLP_{topk_ids[t,k]}(x[t]), written to
        `out` if given (else to the layer's own buffer)."""
        T, K, E, D, I, a = self.T, self.K, self.E, self.D, self.I, self.align
        B.moe_route_permute(topk_ids, topk_w, x, T, K, E, D, a, self.counts, self.offsets,
                            self.perm_src, self.inv_perm, self.w_perm, self.x_perm,
                            self.workspace, stream)
        B.moe_expert_mlp_fwd(self.x_perm, w_gate, w_up, w_down, self.offsets, self._counts(), T,
                             K, E, D, I, a, self.y_perm, self.workspace, stream)
        y = self.y if out is None else out
        B.moe_combine(self.y_perm, self.inv_perm, topk_w, T, K, D, y, stream)
        self._x = x   # the backward gathers its fp16 copy of the sorted rows from x
        return y

    def backward(self, dy, w_gate, w_up, w_down, stream=None, dx_out=None):
        """(dX [T,D] bf16, dW_gate [E,D,I] f32, dW_up [E,D,I] f32, dW_down [E,I,D] f32)
        of L = sum(Y * dy), for the routing of the last forward."""
        T, K, E, D, I, a = self.T, self.K, self.E, self.D, self.I, self.align
        dx = self.dx if dx_out is None else dx_out
        fused = self.reduce_in_backward and T > 0
        B.moe_expert_mlp_bwd(dy, self._x, self.x_perm, self.perm_src, self.w_perm, self.offsets,
                             self._counts(), w_gate, w_up, w_down, T, K, E, D, I, a, self.dx_perm,
                             self.dw_gate, self.dw_up, self.dw_down, self.workspace, stream,
                             inv_perm=self.inv_perm if fused else None, dx=dx if fused else None)
        if not fused:
            B.moe_combine(self.dx_perm, self.inv_perm, None, T, K, D, dx, stream)
        return dx, self.dw_gate, self.dw_up, self.dw_down

    def route(self, logits, router="softmax", stream=None):
        """(topk_ids [T,K] int32, topk_w [T,K] fp32) from router logits [T,E] fp32."""
        T, K, E = self.T, self.K, self.E
        if not hasattr(self, "topk_ids"):
            self.topk_ids = torch.empty(T, K, dtype=torch.int32, device=self.device)
            self.topk_w = torch.empty(T, K, dtype=torch.float32, device=self.device)
        B.moe_router_topk(logits, T, E, K, router, self.topk_ids, self.topk_w, stream)
        self._router = router
        return self.topk_ids, self.topk_w

    def router_backward(self, dy, stream=None):
        """d_logits [T,E] fp32 for the routing of the last route() + forward(): the
        router-weight gradient <dY[t], f_e(x[t])> from the forward's expert outputs,
        then through the router weights to the logits."""
        T, K, E, D = self.T, self.K, self.E, self.D
        if not hasattr(self, "d_topk_w"):
            self.d_topk_w = torch.empty(T, K, dtype=torch.float32, device=self.device)
            self.d_logits = torch.empty(T, E, dtype=torch.float32, device=self.device)
        B.moe_router_weight_grad(dy, self.y_perm, self.inv_perm, T, K, D, self.d_topk_w, stream)
        B.moe_router_backward(self.topk_ids, self.topk_w, self.d_topk_w, T, E, K, self._router,
                              self.d_logits, stream)
        return self.d_logits

    def _counts(self):
        return self.counts if self.skip_padding else None

    def device_error(self, stream=None):
        return B.moe_get_device_error(self.workspace, stream)
