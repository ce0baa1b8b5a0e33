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


class SwiGLUWeights(MLPWeights):
    """Packed per-shard weights of a SwiGLU MLP: W_gate and W_up (h, F) -> one
    [t][2F/t][h] block (tp_pack_swiglu: gate and up rows alternate in groups of
    128), W_down (F, h) -> [t][h][F/t].  No biases on the gate / up side."""

    def __init__(self, W_gate, W_up, W_down, b_down, t):
        h, F = W_up.shape
        assert W_gate.shape == (h, F) and W_down.shape == (F, h) and F % t == 0
        self.h, self.F, self.t = h, F, t
        self.Wup_p = torch.empty(t, 2 * F // t, h, dtype=BF16, device=W_up.device)
        self.Wdown_p = torch.empty(t, h, F // t, dtype=BF16, device=W_up.device)
        L.tp_pack_swiglu(W_gate, W_up, h, F, t, self.Wup_p)
        L.tp_pack_row(W_down, F, h, t, self.Wdown_p)
        self.b_up, self.b_down = None, b_down


def _z_cols(w, act):
    """Columns of a shard's Z / dZ: twice F/t under SwiGLU (gate and up)."""
    return (2 if _act(act) == L.ACT_BY_NAME["swiglu"] else 1) * (w.F // w.t)


def mlp_forward(X, w: MLPWeights, act="gelu_tanh", residual=None, save_z=True, flags=0):
    """Y = sum_i act(X W_up,i + b_up,i) W_down,i + b_down (+ residual).  Returns (Y, Z, A).
    With act="swiglu" (SwiGLUWeights) A_i = silu(X W_gate,i) * (X W_up,i) and Z holds
    the gate and up pre-activations, interleaved as in the packed weights."""
    M = X.shape[0]
    Y = torch.empty(M, w.h, dtype=BF16, device=X.device)
    A = torch.empty(w.t, M, w.F // w.t, dtype=BF16, device=X.device)
    swiglu = _act(act) == L.ACT_BY_NAME["swiglu"]
    Z = torch.empty(w.t, M, _z_cols(w, act), dtype=BF16, device=X.device) if (save_z or swiglu) else None
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
    swiglu = _act(act) == L.ACT_BY_NAME["swiglu"]
    if grads is None:
        grads = {"dWup_p": torch.empty(w.t, _z_cols(w, act), w.h, dtype=torch.float32, device=X.device),
                 "dWdown_p": torch.empty(w.t, w.h, w.F // w.t, dtype=torch.float32, device=X.device),
                 "dbup": None if swiglu else torch.empty(w.F, dtype=torch.float32, device=X.device),
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


# --------------------------------------------------------------------------
# One pre-LN transformer layer: X1 = X + Attn(LN1(X)); Y = X1 + MLP(LN2(X1)).
# With sp=True the LayerNorms and residual adds run on t sequence shards
# ([t][s/t][h], the same bytes as [s][h], so the all-gather entering each TP
# region and the reduce-scatter leaving it are zero-copy) and the LayerNorm
# weight gradients are summed over the shards ("Tensor and sequence
# parallelism", section "Sequence parallelism").  Without SP the LayerNorms are
# replicated: on one GPU that is one LayerNorm over all rows.
# --------------------------------------------------------------------------

class LayerWeights:
    """Packed per-shard weights of one layer (device).  W_qkv is kept in IEEE fp16: the
    layer runs its attention block on an fp16 input (TP_ATTN_F16_INPUT), which the
    softmax of a wide model needs to stay within tolerance."""

    def __init__(self, p, n_heads, head_dim, t):
        d = p["W_qkv"].shape[0]
        F = p["W_up"].shape[1]
        dev = p["W_qkv"].device
        self.d, self.F, self.t, self.n_heads, self.head_dim = d, F, t, n_heads, head_dim
        self.Wqkv_p = torch.empty(t, 3 * d // t, d, dtype=BF16, device=dev)
        self.bqkv_p = torch.empty(t, 3 * d // t, dtype=BF16, device=dev)
        self.Wo_p = torch.empty(t, d, d // t, dtype=BF16, device=dev)
        L.tp_pack_qkv_heads(p["W_qkv"], d, n_heads, head_dim, t, self.Wqkv_p)
        wq16 = torch.empty(t, 3 * d // t, d, dtype=torch.float16, device=dev)
        L.tp_convert_bf16_to_f16(self.Wqkv_p, self.Wqkv_p.numel(), wq16)
        self.Wqkv_p = wq16
        L.tp_pack_qkv_bias(p["b_qkv"], d, n_heads, head_dim, t, self.bqkv_p)
        L.tp_pack_row(p["W_o"], d, d, t, self.Wo_p)
        self.mlp = MLPWeights(p["W_up"], p["b_up"], p["W_down"], p["b_down"], t)
        self.b_o = p["b_o"]
        self.ln1_g, self.ln1_b, self.ln2_g, self.ln2_b = p["ln1_g"], p["ln1_b"], p["ln2_g"], p["ln2_b"]


def layer_forward(X, w: LayerWeights, act="gelu_tanh", causal=True, scale=None, eps=1e-5, sp=False):
    """Returns (Y, saved).  X: [s][h] bf16 ([t][s/t][h] when sp)."""
    s = X.shape[0] if X.dim() == 2 else X.shape[0] * X.shape[1]
    X = X.reshape(s, w.d)
    d, t, dev = w.d, w.t, X.device
    t_ln = t if sp else 1
    scale = (1.0 / w.head_dim ** 0.5) if scale is None else scale
    f32 = torch.float32
    # the attention block's input in IEEE fp16 (TP_ATTN_F16_INPUT)
    Xn1 = torch.empty(s, d, dtype=torch.float16, device=dev)
    m1 = torch.empty(s, dtype=f32, device=dev)
    r1 = torch.empty(s, dtype=f32, device=dev)
    L.tp_sp_layernorm_forward_f16(X, s, d, t_ln, w.ln1_g, w.ln1_b, eps, Xn1, m1, r1)
    X1 = torch.empty(s, d, dtype=BF16, device=dev)
    QKV = torch.empty(t, s, 3 * d // t, dtype=torch.float16, device=dev)  # fp16 attention operands
    O = torch.empty(t, s, d // t, dtype=BF16, device=dev)
    lse = torch.empty(t, w.n_heads // t, s, dtype=f32, device=dev)
    aws = _ws(L.tp_attn_forward_workspace_size(s, d, w.n_heads, w.head_dim, t, 0), dev)  # room for the split-K partials
    L.tp_attn_forward(Xn1, s, d, w.n_heads, w.head_dim, t, int(causal), scale, w.Wqkv_p, w.bqkv_p, w.Wo_p, w.b_o,
                      X, X1, QKV, O, lse, L.TP_ATTN_F16_INPUT, aws, aws.numel())
    Xn2 = torch.empty(s, d, dtype=BF16, device=dev)
    m2 = torch.empty(s, dtype=f32, device=dev)
    r2 = torch.empty(s, dtype=f32, device=dev)
    L.tp_sp_layernorm_forward(X1, s, d, t_ln, w.ln2_g, w.ln2_b, eps, Xn2, m2, r2)
    Y, Z, A = mlp_forward(Xn2, w.mlp, act, residual=X1)
    saved = dict(X=X, Xn1=Xn1, m1=m1, r1=r1, X1=X1, QKV=QKV, O=O, lse=lse, Xn2=Xn2, m2=m2, r2=r2, Z=Z, A=A,
                 s=s, scale=scale, causal=causal, act=act, t_ln=t_ln)
    return Y, saved


def layer_backward(G, saved, w: LayerWeights):
    """Gradients of <Y, G>: dict with dX and every parameter gradient (packed, fp32)."""
    s, d, t, dev = saved["s"], w.d, w.t, G.device
    G = G.reshape(s, d)
    f32 = torch.float32
    g = mlp_backward(G, saved["Xn2"], saved["Z"], saved["A"], w.mlp, saved["act"])
    t_ln = saved["t_ln"]
    dX1 = torch.empty(s, d, dtype=BF16, device=dev)
    ln2 = {k: torch.empty(*shape, dtype=f32, device=dev) for k, shape in
           (("gp", (t_ln, d)), ("bp", (t_ln, d)), ("g", (d,)), ("b", (d,)))}
    L.tp_sp_layernorm_backward(g["dX"], saved["X1"], w.ln2_g, saved["m2"], saved["r2"], G, s, d, t_ln, dX1,
                               ln2["gp"], ln2["bp"], ln2["g"], ln2["b"])
    dXn1 = torch.empty(s, d, dtype=BF16, device=dev)
    dWqkv = torch.empty(t, 3 * d // t, d, dtype=f32, device=dev)
    dbqkv = torch.empty(t, 3 * d // t, dtype=f32, device=dev)
    dWo = torch.empty(t, d, d // t, dtype=f32, device=dev)
    dbo = torch.empty(d, dtype=f32, device=dev)
    nws = L.tp_attn_backward_workspace_size(s, d, w.n_heads, w.head_dim, t, 0)
    ws = _ws(nws, dev)
    L.tp_attn_backward(dX1, saved["Xn1"], saved["QKV"], saved["O"], saved["lse"], s, d, w.n_heads, w.head_dim, t,
                       int(saved["causal"]), saved["scale"], w.Wqkv_p, w.Wo_p, dXn1, dWqkv, dbqkv, dWo, dbo, 0,
                       L.TP_ATTN_F16_INPUT, ws, nws)
    dX = torch.empty(s, d, dtype=BF16, device=dev)
    ln1 = {k: torch.empty(*shape, dtype=f32, device=dev) for k, shape in
           (("gp", (t_ln, d)), ("bp", (t_ln, d)), ("g", (d,)), ("b", (d,)))}
    L.tp_sp_layernorm_backward(dXn1, saved["X"], w.ln1_g, saved["m1"], saved["r1"], dX1, s, d, t_ln, dX,
                               ln1["gp"], ln1["bp"], ln1["g"], ln1["b"])
    return {"dX": dX, "dX1": dX1, "ln1_g": ln1["g"], "ln1_b": ln1["b"], "ln2_g": ln2["g"], "ln2_b": ln2["b"],
            "ln1_g_part": ln1["gp"], "ln2_g_part": ln2["gp"],
            "Wqkv_p": dWqkv, "bqkv_p": dbqkv, "Wo_p": dWo, "b_o": dbo,
            "Wup_p": g["dWup_p"], "b_up": g["dbup"], "Wdown_p": g["dWdown_p"], "b_down": g["dbdown"]}


class DecodeAttnWeights:
    """Packed weights of a TP attention block with grouped-query heads, for
    decode: W_qkv (d, (n_heads + 2 n_kv) head_dim) -> [t][R][d] sharded by KV
    group (replicated KV heads when n_kv < t); W_o (n_heads head_dim, d) ->
    [t][d][n_heads head_dim / t]."""

    def __init__(self, W_qkv, b_qkv, W_o, b_o, n_heads, n_kv, head_dim, t):
        d = W_qkv.shape[0]
        self.d, self.n_heads, self.n_kv, self.head_dim, self.t = d, n_heads, n_kv, head_dim, t
        self.kv_t = n_kv // t if n_kv >= t else 1
        R = (n_heads // t + 2 * self.kv_t) * head_dim
        dev = W_qkv.device
        self.Wqkv_p = torch.empty(t, R, d, dtype=BF16, device=dev)
        L.tp_pack_qkv_gqa(W_qkv, d, n_heads, n_kv, head_dim, t, self.Wqkv_p)
        self.bqkv_p = None
        if b_qkv is not None:
            self.bqkv_p = torch.empty(t, R, dtype=BF16, device=dev)
            L.tp_pack_qkv_gqa_bias(b_qkv, n_heads, n_kv, head_dim, t, self.bqkv_p)
        nq = n_heads * head_dim
        self.Wo_p = torch.empty(t, d, nq // t, dtype=BF16, device=dev)
        L.tp_pack_row(W_o, nq, d, t, self.Wo_p)
        self.b_o = b_o

    def cache_shape(self, B, L_max):
        """Per-shard KV cache [t][kv_t][B][L_max][head_dim] (fp16)."""
        return (self.t, self.kv_t, B, L_max, self.head_dim)

    def workspace(self, B, L_max, device):
        return _ws(L.tp_decode_attn_workspace_size(B, self.d, self.n_heads, self.n_kv, self.head_dim, self.t, L_max),
                   device)


def decode_attn_forward(x, w: DecodeAttnWeights, K_cache, V_cache, pos, scale=None, ws=None, out=None):
    """One decode step: appends each sequence's new key/value at pos[b] in
    every shard's cache copy and returns y [B][d] = sum_i O_i W_o,i + b_o.
    Allocates nothing when ws and out are given (so it can be captured in a
    CUDA graph)."""
    B = x.shape[0]
    L_max = K_cache.shape[3]
    assert K_cache.dtype == torch.float16 and V_cache.dtype == torch.float16 and pos.dtype == torch.int32
    if scale is None:
        scale = w.head_dim ** -0.5
    if ws is None:
        ws = w.workspace(B, L_max, x.device)
    y = out if out is not None else torch.empty(B, w.d, dtype=BF16, device=x.device)
    L.tp_decode_attn_forward(x, B, w.d, w.n_heads, w.n_kv, w.head_dim, w.t, scale, w.Wqkv_p, w.bqkv_p, w.Wo_p,
                             w.b_o, K_cache, V_cache, L_max, pos, y, ws, ws.numel())
    return y
