"""Thin PyTorch-facing layer over the C ABI: torch allocates device memory and
provides the stream; every step of the TP block runs in libtpshard.so.

The f / g operators of "Tensor and sequence parallelism" (section "How
Megatron partitions") are not separate calls here: with the t ranks resident
on one GPU, f's backward all-reduce and g's forward all-reduce are fixed-order
reductions fused into the row-parallel GEMMs, and the identities are just the
same buffer read by every shard.  :class:`TPMLPFunction` exposes the block as
one autograd Function whose forward is "f, column-parallel, act,
row-parallel, g" and whose backward is the mirror image.
"""

from __future__ import annotations

import torch

from . import _lib as L

BF16 = torch.bfloat16


def _act(act):
    return L.ACT_BY_NAME[act] if isinstance(act, str) else int(act)


def _ws(nbytes, device):
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


class MLPWeights:
    """Packed per-shard weights of one TP MLP: W_up (h, F) -> [t][F/t][h],
    W_down (F, h) -> [t][h][F/t]; biases stay as given (b_up is split by the
    same contiguous column blocks)."""

    def __init__(self, W_up, b_up, W_down, b_down, t):
        h, F = W_up.shape
        assert W_down.shape == (F, h) and F % t == 0
        self.h, self.F, self.t = h, F, t
        self.Wup_p = torch.empty(t, F // t, h, dtype=BF16, device=W_up.device)
        self.Wdown_p = torch.empty(t, h, F // t, dtype=BF16, device=W_up.device)
        L.tp_pack_col(W_up, h, F, t, self.Wup_p)
        L.tp_pack_row(W_down, F, h, t, self.Wdown_p)
        self.b_up, self.b_down = b_up, b_down


def mlp_forward(X, w: MLPWeights, act="gelu_tanh", residual=None, save_z=True, flags=0):
    """Y = sum_i act(X W_up,i + b_up,i) W_down,i + b_down (+ residual).  Returns (Y, Z, A)."""
    M = X.shape[0]
    Y = torch.empty(M, w.h, dtype=BF16, device=X.device)
    A = torch.empty(w.t, M, w.F // w.t, dtype=BF16, device=X.device)
    Z = torch.empty_like(A) if save_z else None
    nws = L.tp_mlp_workspace_size(M, w.h, w.F, w.t, flags)
    ws = _ws(nws, X.device)
    L.tp_mlp_forward(X, M, w.h, w.F, w.t, _act(act), w.Wup_p, w.b_up, w.Wdown_p, w.b_down, residual, Y, Z, A,
                     flags, ws, ws.numel())
    return Y, Z, A


def mlp_backward(dY, X, Z, A, w: MLPWeights, act="gelu_tanh", flags=0, grads=None):
    """Gradients of <Y, dY>.  Returns dict dX, dWup_p, dWdown_p, dbup, dbdown
    (weight grads in the packed layouts, fp32).  Pass `grads` to accumulate."""
    M = X.shape[0]
    acc = grads is not None
    if grads is None:
        grads = {"dWup_p": torch.empty(w.t, w.F // w.t, w.h, dtype=torch.float32, device=X.device),
                 "dWdown_p": torch.empty(w.t, w.h, w.F // w.t, dtype=torch.float32, device=X.device),
                 "dbup": torch.empty(w.F, dtype=torch.float32, device=X.device),
                 "dbdown": torch.empty(w.h, dtype=torch.float32, device=X.device)}
    dX = torch.empty(M, w.h, dtype=BF16, device=X.device)
    ws = _ws(L.tp_mlp_backward_workspace_size(M, w.h, w.F, w.t, flags), X.device)
    L.tp_mlp_backward(dY, X, Z, A, M, w.h, w.F, w.t, _act(act), w.Wup_p, w.Wdown_p, dX, grads["dWup_p"],
                      grads["dWdown_p"], grads["dbup"], grads["dbdown"], int(acc), flags, ws, ws.numel())
    out = dict(grads)
    out["dX"] = dX
    return out


class TPMLPFunction(torch.autograd.Function):
    """Autograd wrapper: forward = f (identity) -> column-parallel -> act ->
    row-parallel -> g (fused reduction, bias once); backward = g (identity) ->
    per-shard dgrad / wgrad -> f (fused reduction of the partial dX).
    Weight gradients land in ``weights.grads`` (packed, fp32, accumulated)."""

    @staticmethod
    def forward(ctx, X, weights: MLPWeights, act):
        Y, Z, A = mlp_forward(X.contiguous(), weights, act)
        ctx.save_for_backward(X, Z, A)
        ctx.weights, ctx.act = weights, act
        return Y

    @staticmethod
    def backward(ctx, dY):
        X, Z, A = ctx.saved_tensors
        w = ctx.weights
        prev = getattr(w, "grads", None)
        g = mlp_backward(dY.contiguous(), X, Z, A, w, ctx.act, grads=prev)
        w.grads = {k: g[k] for k in ("dWup_p", "dWdown_p", "dbup", "dbdown")}
        return g["dX"], None, None
