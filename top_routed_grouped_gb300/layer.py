"""``MoELayer``: the layer as a torch module, forward and backward through the C ABI.

RL-Kernel PR #557 "EP4 distributed logprob parity", embedded #503 commit
message, bullets "Routing", "Experts", "Combine" and "Backward": one MoE layer
(top-k routed SwiGLU experts plus a sigmoid-gated shared expert) whose
forward is ``moe_forward`` and whose backward is ``moe_backward``.  This file
only marshals: ``MoEFunction`` is a ``torch.autograd.Function`` that calls the
two entry points on ``torch.cuda.current_stream()`` and hands their outputs
to autograd.  Every step runs in the library's CUDA kernels.

Gradients: the library returns every weight gradient in FP32 (``dW`` is
overwritten, not accumulated).  Autograd casts a gradient to its
parameter's dtype, so a bf16 parameter receives the FP32 gradient rounded
once to bf16 (the FP32 router weight receives it unrounded); dx is the
library's bf16 dx bit for bit.  The routes are held fixed in the backward
(the top-k selection is piecewise constant), as in ``moe_backward``.

Workspaces are caller-visible: pass ``ws_forward`` / ``ws_backward`` (uint8
device tensors of at least ``moe_workspace_size`` bytes) to ``forward``, or
let the layer keep one pair, grown to the largest token count seen
(``MoELayer.workspace``).  A workspace is scratch only: the tensors saved for
the backward are allocated per call, so several forwards may run before
their backwards (gradient accumulation) on the layer's one pair, in stream
order.
"""
from __future__ import annotations

import torch

from . import (backward, dims_of, forward, moe_workspace_size)

_WKEYS = ("w_router", "w_shared_gate", "w_gate_up", "w_down", "ws_gate_up", "ws_down")
_ROUTING = ("topk_ids", "topk_w", "shared_sig", "expert_offsets", "sorted_route", "route_pos", "y_routed", "y_shared")
_SAVED = ("gu", "h", "gu_shared", "h_shared")


class MoEFunction(torch.autograd.Function):
    """y = MoE(x) with the six layer weights as differentiable inputs.

    Inputs: x [T, H]; w_router [E, H] float32; w_shared_gate [H];
    w_gate_up [E, 2I, H]; w_down [E, H, I]; ws_gate_up [2Is, H];
    ws_down [H, Is] (x and the expert weights share one dtype, float32 or
    bfloat16); k; router_bias [E] float32 or None (an input, no gradient);
    ws_fwd / ws_bwd: the two workspaces or None (allocated per call)."""

    @staticmethod
    def forward(ctx, x, w_router, w_shared_gate, w_gate_up, w_down, ws_gate_up, ws_down, k, router_bias=None,
                ws_fwd=None, ws_bwd=None):
        x = x.contiguous()
        stream = torch.cuda.current_stream(x.device)
        f = forward(x, w_router, w_shared_gate, w_gate_up, w_down, ws_gate_up, ws_down, int(k),
                    router_bias=router_bias, save_for_backward=True, stream=stream, ws=ws_fwd)
        ctx.save_for_backward(x, w_router, w_shared_gate, w_gate_up, w_down, ws_gate_up, ws_down,
                              *[f[n] for n in _ROUTING], *[f["saved"][n] for n in _SAVED])
        ctx.ws_bwd = ws_bwd
        ctx.mark_non_differentiable(*[f[n] for n in ("topk_ids", "topk_w", "shared_sig")])
        return f["y"], f["topk_ids"], f["topk_w"], f["shared_sig"]

    @staticmethod
    def backward(ctx, dy, _d_ids=None, _d_w=None, _d_sig=None):
        t = ctx.saved_tensors
        x, weights = t[0], t[1:7]
        fwd = dict(zip(_ROUTING, t[7:7 + len(_ROUTING)]))
        fwd["saved"] = dict(zip(_SAVED, t[7 + len(_ROUTING):]))
        if dy is None:
            dy = torch.zeros_like(x)
        g = backward(fwd, dy.contiguous(), x, *weights, ws=ctx.ws_bwd,
                     stream=torch.cuda.current_stream(x.device))
        return (g["dx"], g["dw_router"], g["dw_shared_gate"], g["dw_gate_up"], g["dw_down"], g["dws_gate_up"],
                g["dws_down"], None, None, None, None)


class MoELayer(torch.nn.Module):
    """One MoE layer: E routed SwiGLU experts (top-k) plus a sigmoid-gated
    shared SwiGLU expert, forward ``moe_forward``, backward ``moe_backward``.

    Parameters (the library's layout, ``nn.Linear`` [out, in] rows):
    ``w_router`` [E, H] float32, ``w_shared_gate`` [H], ``w_gate_up``
    [E, 2I, H] (I gate rows, then I up rows), ``w_down`` [E, H, I],
    ``ws_gate_up`` [2Is, H], ``ws_down`` [H, Is]; ``dtype`` bfloat16 or
    float32 for all but the router.  ``router_bias`` (optional [E] float32
    buffer) is added to the logits and gets no gradient.

    ``forward(x)`` returns y [T, H]; ``last_routes`` holds the step's
    topk_ids [T, k], topk_w [T, k] and shared_sig [T] (no gradient)."""

    def __init__(self, hidden: int, n_experts: int, top_k: int, intermediate: int, shared_intermediate: int,
                 dtype: torch.dtype = torch.bfloat16, device=None, router_bias: torch.Tensor | None = None,
                 init_std: float = 0.02):
        super().__init__()
        H, E, I_, Is = hidden, n_experts, intermediate, shared_intermediate
        dev = torch.device("cuda") if device is None else torch.device(device)
        self.top_k = int(top_k)
        mk = lambda *shape, dt=dtype: torch.nn.Parameter(  # noqa: E731
            torch.empty(*shape, dtype=dt, device=dev).normal_(0.0, init_std))
        self.w_router = mk(E, H, dt=torch.float32)
        self.w_shared_gate = mk(H)
        self.w_gate_up = mk(E, 2 * I_, H)
        self.w_down = mk(E, H, I_)
        self.ws_gate_up = mk(2 * Is, H)
        self.ws_down = mk(H, Is)
        self.register_buffer("router_bias", None if router_bias is None else
                             router_bias.to(device=dev, dtype=torch.float32))
        self._ws: tuple[torch.Tensor, torch.Tensor] | None = None
        self.last_routes: dict = {}

    def weights(self):
        return tuple(getattr(self, n) for n in _WKEYS)

    def workspace(self, T: int) -> tuple[torch.Tensor, torch.Tensor]:
        """The forward and backward workspaces for T tokens: the layer's one
        pair, reallocated only when T needs more bytes than it holds."""
        d = dims_of(torch.empty(T, self.w_router.shape[1], dtype=self.w_gate_up.dtype, device="meta"),
                    self.w_router, self.w_gate_up, self.ws_gate_up, self.top_k)
        need = [max(moe_workspace_size(d, op), 256) for op in ("forward", "backward")]
        if self._ws is None or any(w.numel() < n for w, n in zip(self._ws, need)):
            old = (0, 0) if self._ws is None else tuple(w.numel() for w in self._ws)
            self._ws = tuple(torch.empty(max(n, o), dtype=torch.uint8, device=self.w_router.device)
                             for n, o in zip(need, old))
        return self._ws

    def forward(self, x: torch.Tensor, ws_forward: torch.Tensor | None = None,
                ws_backward: torch.Tensor | None = None) -> torch.Tensor:
        if ws_forward is None or ws_backward is None:
            wf, wb = self.workspace(x.shape[0])
            ws_forward = wf if ws_forward is None else ws_forward
            ws_backward = wb if ws_backward is None else ws_backward
        y, ids, w, sig = MoEFunction.apply(x, *self.weights(), self.top_k, self.router_bias, ws_forward, ws_backward)
        self.last_routes = {"topk_ids": ids, "topk_w": w, "shared_sig": sig}
        return y
