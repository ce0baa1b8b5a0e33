"""fp64 oracle: unsplit and t-way sharded Megatron TP block (test infrastructure only).

Notation follows "02 — Tensor Parallelism" (project-fortress roadmap, section
"Column-parallel vs row-parallel — the derivation"): activations multiply
weights from the left, ``Y = X @ W`` with W stored (in, out).  The hidden
dimension of the MLP is split into t contiguous column blocks
``C_i = [i*F/t, (i+1)*F/t)`` in rank order, as the ``cols = slice(rank*FFN//tp,
(rank+1)*FFN//tp)`` line of "Tensor and sequence parallelism" (ai-infra
handbooks, section "The implementation", tp_mlp_check.py) and the
``for columns in ((0, 1), (2, 3))`` loop of "Tensor Parallelism's Communication
Boundary" (section "Run the example") do.

Every routine takes float64 numpy arrays (use :func:`bf16_to_f64` on the seeded
bf16 bits first) and returns float64 results; no intermediate is rounded.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "bf16_to_f64", "f64_to_bf16_bits", "shard_slice",
    "pack_col_weight", "pack_row_weight", "pack_swiglu_weight", "pack_qkv_weight",
    "pack_qkv_bias", "qkv_shard_columns", "unpack_col_weight", "unpack_row_weight",
    "ACTIVATIONS", "act", "act_grad", "silu", "silu_grad",
    "mlp_forward_unsplit", "mlp_forward_sharded", "mlp_backward_unsplit", "mlp_backward_sharded",
    "swiglu_forward_unsplit", "swiglu_forward_sharded", "swiglu_backward_sharded",
    "mlp_forward_rowfirst_split", "mlp_forward_bias_every_shard", "mlp_fg_swapped",
    "attention_head_forward", "attention_head_backward",
    "attn_forward_unsplit", "attn_forward_sharded", "attn_backward_unsplit", "attn_backward_sharded",
    "layernorm_forward", "layernorm_backward", "sp_layernorm_forward", "sp_layernorm_backward",
    "all_gather_seq", "reduce_scatter_seq",
    "layer_forward", "layer_backward", "layer_forward_rows",
    "expanded_tensor_bytes", "reduction_tensor_bytes", "allreduce_payload_bytes",
    "mlp_fwd_bwd_flops",
]


# ---------------------------------------------------------------------------
# bf16 <-> float64.  bf16 is the top half of an IEEE binary32.
# ---------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of raw bf16 bit patterns (uint16) as float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 to bf16 bits, round-to-nearest-even (via binary32 first).

    Diagnostic helper only (a "mirror" of the GPU's storage points); parity is
    judged against the unrounded fp64 results.
    """
    f = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = (f & 0x7FFFFFFF) > 0x7F800000
    lsb = (f >> 16) & 1
    r = ((f + 0x7FFF + lsb) >> 16).astype(np.uint16)
    r[nan] = 0x7FC0
    return r


# ---------------------------------------------------------------------------
# Shard layout.  Column-parallel: W (in, out) split along the output dim;
# row-parallel: W split along the input dim ("02 — Tensor Parallelism",
# sections "Column-parallel" and "Row-parallel").  Packed per-shard slices are
# stored (out, in) -- the per-rank ``F.linear`` weights of tp_mlp_check.py in
# "Tensor and sequence parallelism", ``w1[cols]`` and ``w2[:, cols]``.
# These work on any dtype (the tests pass raw bf16 bit patterns).
# ---------------------------------------------------------------------------

def shard_slice(n: int, t: int, i: int) -> slice:
    """Rows/columns owned by shard i: [i*n/t, (i+1)*n/t) (t must divide n)."""
    assert n % t == 0, "t must divide the split dimension"
    return slice(i * n // t, (i + 1) * n // t)


def pack_col_weight(W: np.ndarray, t: int) -> np.ndarray:
    """W (h, F) -> [t][F/t][h]: shard i holds W[:, C_i] stored transposed."""
    h, F = W.shape
    return np.stack([W[:, shard_slice(F, t, i)].T for i in range(t)])


def unpack_col_weight(Wp: np.ndarray) -> np.ndarray:
    t, Ft, h = Wp.shape
    return np.concatenate([Wp[i].T for i in range(t)], axis=1)


def pack_row_weight(W: np.ndarray, t: int) -> np.ndarray:
    """W (F, h) -> [t][h][F/t]: shard i holds W[C_i, :] stored transposed."""
    F, h = W.shape
    return np.stack([W[shard_slice(F, t, i), :].T for i in range(t)])


def unpack_row_weight(Wp: np.ndarray) -> np.ndarray:
    t, h, Ft = Wp.shape
    return np.concatenate([Wp[i].T for i in range(t)], axis=0)


def pack_swiglu_weight(Wg: np.ndarray, Wu: np.ndarray, t: int, group: int = 128) -> np.ndarray:
    """Gate and up (h, F) -> [t][F/t/group][2][group][h].

    Shard i takes columns C_i of both matrices (the "(times 2 for SwiGLU)" of
    the up-projection in "02 — Tensor Parallelism", section "The core
    observation"); inside a shard, groups of ``group`` gate rows and the
    matching ``group`` up rows alternate.
    """
    h, F = Wg.shape
    Ft = F // t
    assert Ft % group == 0
    out = []
    for i in range(t):
        cs = shard_slice(F, t, i)
        g_i, u_i = Wg[:, cs].T, Wu[:, cs].T          # (Ft, h) each
        blocks = []
        for q in range(Ft // group):
            rs = slice(q * group, (q + 1) * group)
            blocks.append(np.stack([g_i[rs], u_i[rs]]))
        out.append(np.stack(blocks))
    return np.stack(out)


def qkv_shard_columns(d: int, n_heads: int, head_dim: int, t: int, i: int) -> np.ndarray:
    """Columns of W_qkv (d, 3d), laid out [Q|K|V], owned by shard i.

    Shard i owns heads [i*n_heads/t, (i+1)*n_heads/t) of Q, K and V ("02 —
    Tensor Parallelism", section "The attention pairing"; "Megatron-LM: Tensor
    Parallelism", section "Attention Block").  Order: its Q heads, its K heads,
    its V heads.
    """
    assert n_heads % t == 0 and n_heads * head_dim == d
    hs = shard_slice(n_heads, t, i)
    cols = []
    for part in range(3):
        for j in range(hs.start, hs.stop):
            base = part * d + j * head_dim
            cols.extend(range(base, base + head_dim))
    return np.asarray(cols, dtype=np.int64)


def pack_qkv_weight(Wqkv: np.ndarray, n_heads: int, head_dim: int, t: int) -> np.ndarray:
    """W_qkv (d, 3d) -> [t][3d/t][d]: shard i's columns, stored transposed."""
    d = Wqkv.shape[0]
    return np.stack([Wqkv[:, qkv_shard_columns(d, n_heads, head_dim, t, i)].T for i in range(t)])


def pack_qkv_bias(b: np.ndarray, n_heads: int, head_dim: int, t: int) -> np.ndarray:
    d = b.shape[0] // 3
    return np.stack([b[qkv_shard_columns(d, n_heads, head_dim, t, i)] for i in range(t)])


# ---------------------------------------------------------------------------
# Elementwise activations.  They act coordinate by coordinate, which is why
# they commute with the column split ("02 — Tensor Parallelism", section "The
# MLP pairing"; "Tensor Parallelism's Communication Boundary", section
# "Follow the coordinates").
# GeLU-tanh: Hendrycks & Gimpel's tanh approximation; GeLU-erf: the exact
# form, what ``F.gelu`` computes by default in tp_mlp_check.py.
# ---------------------------------------------------------------------------

_SQRT_2_OVER_PI = math.sqrt(2.0 / math.pi)
_GELU_C = 0.044715


def _erf(x: np.ndarray) -> np.ndarray:
    from scipy.special import erf
    return erf(x)


def act(name: str, z: np.ndarray) -> np.ndarray:
    if name == "identity":
        return z.copy()
    if name == "relu":
        return np.maximum(z, 0.0)
    if name == "gelu_tanh":
        u = _SQRT_2_OVER_PI * (z + _GELU_C * z ** 3)
        return 0.5 * z * (1.0 + np.tanh(u))
    if name == "gelu_erf":
        return 0.5 * z * (1.0 + _erf(z / math.sqrt(2.0)))
    raise ValueError(name)


def act_grad(name: str, z: np.ndarray) -> np.ndarray:
    """d act / d z, the closed-form derivative of each activation."""
    if name == "identity":
        return np.ones_like(z)
    if name == "relu":
        return (z > 0).astype(np.float64)
    if name == "gelu_tanh":
        u = _SQRT_2_OVER_PI * (z + _GELU_C * z ** 3)
        th = np.tanh(u)
        du = _SQRT_2_OVER_PI * (1.0 + 3.0 * _GELU_C * z ** 2)
        return 0.5 * (1.0 + th) + 0.5 * z * (1.0 - th ** 2) * du
    if name == "gelu_erf":
        cdf = 0.5 * (1.0 + _erf(z / math.sqrt(2.0)))
        pdf = np.exp(-0.5 * z ** 2) / math.sqrt(2.0 * math.pi)
        return cdf + z * pdf
    raise ValueError(name)


ACTIVATIONS = ("identity", "relu", "gelu_tanh", "gelu_erf")


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def silu_grad(z: np.ndarray) -> np.ndarray:
    s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


# ---------------------------------------------------------------------------
# TP MLP: column-parallel W_up -> activation -> row-parallel W_down -> g.
# "02 — Tensor Parallelism", section "The MLP pairing"; "Tensor and sequence
# parallelism", section "How Megatron partitions" (the f/g table).
# ---------------------------------------------------------------------------

def _zeros_if_none(b, n):
    return np.zeros(n) if b is None else b


def mlp_forward_unsplit(X, W_up, b_up, W_down, b_down, act_name):
    """Z = X W_up + b_up; A = act(Z); Y = A W_down + b_down."""
    h, F = W_up.shape
    Z = X @ W_up + _zeros_if_none(b_up, F)
    A = act(act_name, Z)
    Y = A @ W_down + _zeros_if_none(b_down, h)
    return {"Z": Z, "A": A, "Y": Y}


def mlp_forward_sharded(X, W_up, b_up, W_down, b_down, act_name, t):
    """The same block as t ranks compute it.

    f forward is the identity: every shard reads the same X.  Shard i computes
    Z_i = X W_up[:, C_i] + b_up[C_i] (its own slice of the column bias),
    A_i = act(Z_i) and the full-shaped partial P_i = A_i W_down[C_i, :].
    g forward is the all-reduce: Y = sum_i P_i, then the output bias once
    ("Tensor Parallelism's Communication Boundary": adding the same output
    bias on every worker before the reduction would duplicate it).
    """
    h, F = W_up.shape
    b_up = _zeros_if_none(b_up, F)
    b_down = _zeros_if_none(b_down, h)
    Zs, As, Ps = [], [], []
    for i in range(t):
        C = shard_slice(F, t, i)
        X_i = X                                   # f: identity forward
        Z_i = X_i @ W_up[:, C] + b_up[C]
        A_i = act(act_name, Z_i)
        P_i = A_i @ W_down[C, :]
        Zs.append(Z_i); As.append(A_i); Ps.append(P_i)
    Y = np.zeros_like(Ps[0])
    for i in range(t):                            # g: all-reduce (sum of partials)
        Y = Y + Ps[i]
    Y = Y + b_down                                # bias once, after the sum
    return {"Z": Zs, "A": As, "P": Ps, "Y": Y}


def mlp_backward_unsplit(G, X, W_up, W_down, Z, A, act_name):
    """Gradients of L = <Y, G> through the unsplit MLP."""
    db_down = G.sum(axis=0)
    dW_down = A.T @ G
    dA = G @ W_down.T
    dZ = dA * act_grad(act_name, Z)
    db_up = dZ.sum(axis=0)
    dW_up = X.T @ dZ
    dX = dZ @ W_up.T
    return {"dX": dX, "dW_up": dW_up, "dW_down": dW_down, "db_up": db_up, "db_down": db_down,
            "dZ": dZ}


def mlp_backward_sharded(G, X, W_up, W_down, fwd, act_name, t, weight_grads=True):
    """Backward as t ranks compute it.

    g backward is the identity: every shard gets G unchanged.  Shard i forms
    dA_i = G W_down[C_i, :]^T, dZ_i = dA_i * act'(Z_i), its own weight grads
    dW_down[C_i, :] = A_i^T G and dW_up[:, C_i] = X^T dZ_i (no communication:
    "Parallelism Strategies #1 - Tensor Parallelism", weight-shard gradients),
    and a partial input grad dX_i = dZ_i W_up[:, C_i]^T.  f backward is the
    all-reduce: dX = sum_i dX_i.  The output-bias grad is taken once.
    weight_grads=False leaves dW_up and dW_down out (zeros): the input grad
    alone, for callers that only follow the gradient through the block.
    """
    h, F = W_up.shape
    dW_up = np.zeros_like(W_up)
    dW_down = np.zeros_like(W_down)
    db_up = np.zeros(F)
    dZs, dXs = [], []
    for i in range(t):
        C = shard_slice(F, t, i)
        G_i = G                                   # g: identity backward
        dA_i = G_i @ W_down[C, :].T
        dZ_i = dA_i * act_grad(act_name, fwd["Z"][i])
        db_up[C] = dZ_i.sum(axis=0)
        if weight_grads:
            dW_down[C, :] = fwd["A"][i].T @ G_i
            dW_up[:, C] = X.T @ dZ_i
        dXs.append(dZ_i @ W_up[:, C].T)
        dZs.append(dZ_i)
    dX = np.zeros_like(dXs[0])
    for i in range(t):                            # f: all-reduce of the partial dX
        dX = dX + dXs[i]
    return {"dX": dX, "dX_partials": dXs, "dW_up": dW_up, "dW_down": dW_down,
            "db_up": db_up, "db_down": G.sum(axis=0), "dZ": dZs}


# SwiGLU: A = silu(X W_gate) * (X W_up); gate and up are both column-split
# with the same C_i, so the product stays local to the shard.

def swiglu_forward_unsplit(X, W_gate, W_up, W_down):
    Zg = X @ W_gate
    Zu = X @ W_up
    A = silu(Zg) * Zu
    return {"Zg": Zg, "Zu": Zu, "A": A, "Y": A @ W_down}


def swiglu_forward_sharded(X, W_gate, W_up, W_down, t):
    h, F = W_up.shape
    Zg, Zu, As, Ps = [], [], [], []
    for i in range(t):
        C = shard_slice(F, t, i)
        g = X @ W_gate[:, C]
        u = X @ W_up[:, C]
        a = silu(g) * u
        Zg.append(g); Zu.append(u); As.append(a)
        Ps.append(a @ W_down[C, :])
    Y = np.zeros_like(Ps[0])
    for i in range(t):
        Y = Y + Ps[i]
    return {"Zg": Zg, "Zu": Zu, "A": As, "P": Ps, "Y": Y}


def swiglu_backward_sharded(G, X, W_gate, W_up, W_down, fwd, t):
    h, F = W_up.shape
    dWg = np.zeros_like(W_gate); dWu = np.zeros_like(W_up); dWd = np.zeros_like(W_down)
    dX = np.zeros_like(X)
    for i in range(t):
        C = shard_slice(F, t, i)
        g, u = fwd["Zg"][i], fwd["Zu"][i]
        dA = G @ W_down[C, :].T
        dg = dA * u * silu_grad(g)
        du = dA * silu(g)
        dWd[C, :] = fwd["A"][i].T @ G
        dWg[:, C] = X.T @ dg
        dWu[:, C] = X.T @ du
        dX = dX + (dg @ W_gate[:, C].T + du @ W_up[:, C].T)
    return {"dX": dX, "dW_gate": dWg, "dW_up": dWu, "dW_down": dWd}


# --- deliberately wrong variants (negative pins) ----------------------------

def mlp_forward_rowfirst_split(X, W_up, b_up, W_down, b_down, act_name, t):
    """WRONG on purpose: split W_up along its *input* dim and apply the
    activation to each worker's partial pre-activation before combining.

    "Tensor Parallelism's Communication Boundary" (section "Count the object,
    then the collective") explains why this fails: act(a+b) != act(a)+act(b).
    """
    h, F = W_up.shape
    b_up = _zeros_if_none(b_up, F)
    hidden = np.zeros((X.shape[0], F))
    for i in range(t):
        R = shard_slice(h, t, i)
        part = X[:, R] @ W_up[R, :] + (b_up if i == 0 else 0.0)
        hidden = hidden + act(act_name, part)
    return hidden @ W_down + _zeros_if_none(b_down, W_down.shape[1])


def mlp_forward_bias_every_shard(X, W_up, b_up, W_down, b_down, act_name, t):
    """WRONG on purpose: every shard adds the output bias before the sum."""
    r = mlp_forward_sharded(X, W_up, b_up, W_down, None, act_name, t)
    Y = np.zeros_like(r["Y"])
    for i in range(t):
        Y = Y + (r["P"][i] + b_down)
    return Y


def mlp_fg_swapped(X, W_up, b_up, W_down, b_down, act_name, t, G):
    """WRONG on purpose: g at the entry and f at the exit of the TP region.

    Per "Tensor and sequence parallelism" (Exercises, question 2): the entry
    all-reduce sums t identical inputs (X becomes t*X), the exit no longer sums
    the partials, and backward never sums the partial input grads.  Returns
    rank 0's output and rank 0's input grad.
    """
    h, F = W_up.shape
    X_in = np.zeros_like(X)
    for _ in range(t):                             # g forward at the entry: all-reduce
        X_in = X_in + X
    C = shard_slice(F, t, 0)
    Z0 = X_in @ W_up[:, C] + _zeros_if_none(b_up, F)[C]
    A0 = act(act_name, Z0)
    out0 = A0 @ W_down[C, :] + _zeros_if_none(b_down, h)   # f forward at the exit: identity
    G_in = np.zeros_like(G)
    for _ in range(t):                             # f backward at the exit: all-reduce
        G_in = G_in + G
    dZ0 = (G_in @ W_down[C, :].T) * act_grad(act_name, Z0)
    dX0 = dZ0 @ W_up[:, C].T                       # g backward at the entry: identity
    return out0, dX0


# ---------------------------------------------------------------------------
# Attention, sharded by head.  "Megatron-LM: Tensor Parallelism", section
# "The Transformer Layer Partitioning": S = Q K^T, P = softmax(S), O = P V,
# Output = O W_O.  The scale factor and the causal mask are parameters (the
# page shows neither); the reading taken is scale = 1/sqrt(head_dim), causal.
# ---------------------------------------------------------------------------

def attention_head_forward(Q, K, V, causal, scale):
    """One head: S = scale * Q K^T, masked where key > query, row softmax, O = P V.

    Returns O, P and the log-sum-exp of each scaled, masked score row.
    """
    N = Q.shape[0]
    S = scale * (Q @ K.T)
    if causal:
        mask = np.triu(np.ones((N, K.shape[0]), dtype=bool), k=1)
        S = np.where(mask, -np.inf, S)
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    den = E.sum(axis=1, keepdims=True)
    P = E / den
    lse = (m + np.log(den))[:, 0]
    return P @ V, P, lse


def attention_head_backward(dO, Q, K, V, P, scale):
    """Softmax-attention backward for one head (masked entries have P = 0)."""
    dV = P.T @ dO
    dP = dO @ V.T
    dS = P * (dP - (dP * P).sum(axis=1, keepdims=True))
    dQ = scale * (dS @ K)
    dK = scale * (dS.T @ Q)
    return dQ, dK, dV


def _head_cols(part, j, d, head_dim):
    base = part * d + j * head_dim
    return slice(base, base + head_dim)


def attn_forward_unsplit(Xn, W_qkv, b_qkv, W_o, b_o, n_heads, head_dim, causal, scale):
    N, d = Xn.shape
    QKV = Xn @ W_qkv + _zeros_if_none(b_qkv, 3 * d)
    O = np.zeros((N, d))
    Ps, lses = [], []
    for j in range(n_heads):
        Q = QKV[:, _head_cols(0, j, d, head_dim)]
        K = QKV[:, _head_cols(1, j, d, head_dim)]
        V = QKV[:, _head_cols(2, j, d, head_dim)]
        o, p, lse = attention_head_forward(Q, K, V, causal, scale)
        O[:, j * head_dim:(j + 1) * head_dim] = o
        Ps.append(p); lses.append(lse)
    Y = O @ W_o + _zeros_if_none(b_o, d)
    return {"QKV": QKV, "O": O, "P": Ps, "lse": np.stack(lses), "Y": Y}


def attn_forward_sharded(Xn, W_qkv, b_qkv, W_o, b_o, n_heads, head_dim, causal, scale, t):
    """Shard i: column-parallel W_qkv on its heads (f forward = identity),
    attention on its heads only, row-parallel W_o on the matching rows; then g
    sums the t partials and the output bias is added once."""
    N, d = Xn.shape
    b_qkv = _zeros_if_none(b_qkv, 3 * d)
    hpr = n_heads // t
    dt = d // t
    QKVs, Os, Ps_attn, lses, partials = [], [], [], [], []
    for i in range(t):
        cols = qkv_shard_columns(d, n_heads, head_dim, t, i)
        QKV_i = Xn @ W_qkv[:, cols] + b_qkv[cols]          # [N][3d/t] = [Q_i|K_i|V_i]
        O_i = np.zeros((N, dt))
        for jj in range(hpr):
            hs = slice(jj * head_dim, (jj + 1) * head_dim)
            Q = QKV_i[:, 0 * dt:1 * dt][:, hs]
            K = QKV_i[:, 1 * dt:2 * dt][:, hs]
            V = QKV_i[:, 2 * dt:3 * dt][:, hs]
            o, p, lse = attention_head_forward(Q, K, V, causal, scale)
            O_i[:, hs] = o
            Ps_attn.append(p); lses.append(lse)
        rows = shard_slice(d, t, i)
        partials.append(O_i @ W_o[rows, :])
        QKVs.append(QKV_i); Os.append(O_i)
    Y = np.zeros((N, d))
    for i in range(t):
        Y = Y + partials[i]
    Y = Y + _zeros_if_none(b_o, d)
    return {"QKV": QKVs, "O": Os, "P": Ps_attn, "lse": np.stack(lses), "partials": partials, "Y": Y}


def attn_backward_unsplit(G, Xn, W_qkv, W_o, fwd, n_heads, head_dim, scale):
    N, d = Xn.shape
    dW_o = fwd["O"].T @ G
    db_o = G.sum(axis=0)
    dO = G @ W_o.T
    QKV = fwd["QKV"]
    dQKV = np.zeros_like(QKV)
    for j in range(n_heads):
        cq, ck, cv = (_head_cols(p, j, d, head_dim) for p in range(3))
        dq, dk, dv = attention_head_backward(dO[:, j * head_dim:(j + 1) * head_dim],
                                             QKV[:, cq], QKV[:, ck], QKV[:, cv], fwd["P"][j], scale)
        dQKV[:, cq] = dq; dQKV[:, ck] = dk; dQKV[:, cv] = dv
    return {"dXn": dQKV @ W_qkv.T, "dW_qkv": Xn.T @ dQKV, "db_qkv": dQKV.sum(axis=0),
            "dW_o": dW_o, "db_o": db_o, "dQKV": dQKV}


def attn_backward_sharded(G, Xn, W_qkv, W_o, fwd, n_heads, head_dim, scale, t):
    """g backward identity (G to every shard); per shard dO_i = G W_o[rows_i]^T,
    head-local softmax backward, dQKV_i; per-shard weight grads; f backward:
    dXn = sum_i dQKV_i W_qkv[:, cols_i]^T."""
    N, d = Xn.shape
    hpr = n_heads // t
    dt = d // t
    dW_qkv = np.zeros_like(W_qkv)
    dW_o = np.zeros_like(W_o)
    db_qkv = np.zeros(3 * d)
    dXn_parts, dQKVs = [], []
    for i in range(t):
        cols = qkv_shard_columns(d, n_heads, head_dim, t, i)
        rows = shard_slice(d, t, i)
        dO_i = G @ W_o[rows, :].T
        dW_o[rows, :] = fwd["O"][i].T @ G
        QKV_i = fwd["QKV"][i]
        dQKV_i = np.zeros_like(QKV_i)
        for jj in range(hpr):
            hs = slice(jj * head_dim, (jj + 1) * head_dim)
            sq = slice(0 * dt + hs.start, 0 * dt + hs.stop)
            sk = slice(1 * dt + hs.start, 1 * dt + hs.stop)
            sv = slice(2 * dt + hs.start, 2 * dt + hs.stop)
            dq, dk, dv = attention_head_backward(dO_i[:, hs], QKV_i[:, sq], QKV_i[:, sk], QKV_i[:, sv],
                                                 fwd["P"][i * hpr + jj], scale)
            dQKV_i[:, sq] = dq; dQKV_i[:, sk] = dk; dQKV_i[:, sv] = dv
        dW_qkv[:, cols] = Xn.T @ dQKV_i
        db_qkv[cols] = dQKV_i.sum(axis=0)
        dXn_parts.append(dQKV_i @ W_qkv[:, cols].T)
        dQKVs.append(dQKV_i)
    dXn = np.zeros_like(Xn)
    for i in range(t):
        dXn = dXn + dXn_parts[i]
    return {"dXn": dXn, "dXn_partials": dXn_parts, "dW_qkv": dW_qkv, "db_qkv": db_qkv,
            "dW_o": dW_o, "db_o": G.sum(axis=0), "dQKV": dQKVs}


# ---------------------------------------------------------------------------
# LayerNorm and the sequence-parallel region ("Tensor and sequence
# parallelism", section "Sequence parallelism"; "02 — Tensor Parallelism",
# section "Sequence parallelism (Megatron-3)").  Biased variance, eps inside
# the square root, affine gamma and beta.
# ---------------------------------------------------------------------------

def layernorm_forward(x, gamma, beta, eps):
    mean = x.mean(axis=1)
    var = ((x - mean[:, None]) ** 2).mean(axis=1)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mean[:, None]) * rstd[:, None]
    return xhat * gamma + beta, mean, rstd


def layernorm_backward(dy, x, gamma, mean, rstd):
    h = x.shape[1]
    xhat = (x - mean[:, None]) * rstd[:, None]
    dgamma = (dy * xhat).sum(axis=0)
    dbeta = dy.sum(axis=0)
    g = dy * gamma
    dx = rstd[:, None] * (g - g.sum(axis=1, keepdims=True) / h
                          - xhat * (g * xhat).sum(axis=1, keepdims=True) / h)
    return dx, dgamma, dbeta


def sp_layernorm_forward(X_sh, gamma, beta, eps):
    """X_sh [t][s/t][h]: each shard normalises only its own s/t rows."""
    ys, means, rstds = [], [], []
    for j in range(X_sh.shape[0]):
        y, m, r = layernorm_forward(X_sh[j], gamma, beta, eps)
        ys.append(y); means.append(m); rstds.append(r)
    return np.stack(ys), np.stack(means), np.stack(rstds)


def sp_layernorm_backward(dY_sh, X_sh, gamma, mean, rstd):
    """Per-shard dX rows and partial (dgamma_j, dbeta_j); the weight grads are
    then summed over the shards -- the extra all-reduce of the LayerNorm weight
    gradient that sequence parallelism needs."""
    t = X_sh.shape[0]
    dxs, dgp, dbp = [], [], []
    for j in range(t):
        dx, dg, db = layernorm_backward(dY_sh[j], X_sh[j], gamma, mean[j], rstd[j])
        dxs.append(dx); dgp.append(dg); dbp.append(db)
    dgamma = np.zeros_like(gamma); dbeta = np.zeros_like(gamma)
    for j in range(t):
        dgamma = dgamma + dgp[j]
        dbeta = dbeta + dbp[j]
    return np.stack(dxs), np.stack(dgp), np.stack(dbp), dgamma, dbeta


def all_gather_seq(shards):
    """GatherSeq forward: concatenate the sequence shards along rows."""
    return np.concatenate(list(shards), axis=0)


def reduce_scatter_seq(partials, t):
    """ScatterSeq forward: sum the t full-shaped partials, then rank j keeps
    rows [j*s/t, (j+1)*s/t)."""
    tot = np.zeros_like(partials[0])
    for p in partials:
        tot = tot + p
    s = tot.shape[0]
    return np.stack([tot[shard_slice(s, t, j)] for j in range(t)])


# ---------------------------------------------------------------------------
# One pre-LN transformer layer: X1 = X + Attn(LN1(X)); Y = X1 + MLP(LN2(X1)).
# With sp=True the LayerNorms and residual adds run on sequence shards and the
# TP regions are entered with an all-gather and left with a reduce-scatter.
# ---------------------------------------------------------------------------

def layer_forward(X, p, cfg, t, sp=False):
    """X: [s][h] (sp=False) or [t][s/t][h] (sp=True).  p: dict of float64
    parameters in unpacked (in, out) form: ln1_g, ln1_b, W_qkv, b_qkv, W_o, b_o,
    ln2_g, ln2_b, W_up, b_up, W_down, b_down.  cfg: n_heads, head_dim, causal,
    scale, eps, act."""
    nh, dh, eps = cfg["n_heads"], cfg["head_dim"], cfg["eps"]
    if not sp:
        Xn1, m1, r1 = layernorm_forward(X, p["ln1_g"], p["ln1_b"], eps)
        at = attn_forward_sharded(Xn1, p["W_qkv"], p["b_qkv"], p["W_o"], p["b_o"], nh, dh,
                                  cfg["causal"], cfg["scale"], t)
        X1 = X + at["Y"]
        Xn2, m2, r2 = layernorm_forward(X1, p["ln2_g"], p["ln2_b"], eps)
        ml = mlp_forward_sharded(Xn2, p["W_up"], p["b_up"], p["W_down"], p["b_down"], cfg["act"], t)
        Y = X1 + ml["Y"]
        return {"Xn1": Xn1, "m1": m1, "r1": r1, "attn": at, "X1": X1, "Xn2": Xn2, "m2": m2,
                "r2": r2, "mlp": ml, "Y": Y}
    Xn1_sh, m1, r1 = sp_layernorm_forward(X, p["ln1_g"], p["ln1_b"], eps)
    Xn1 = all_gather_seq(Xn1_sh)
    at = attn_forward_sharded(Xn1, p["W_qkv"], p["b_qkv"], p["W_o"], None, nh, dh,
                              cfg["causal"], cfg["scale"], t)
    X1_sh = reduce_scatter_seq(at["partials"], t) + _zeros_if_none(p["b_o"], X.shape[2]) + X
    Xn2_sh, m2, r2 = sp_layernorm_forward(X1_sh, p["ln2_g"], p["ln2_b"], eps)
    Xn2 = all_gather_seq(Xn2_sh)
    ml = mlp_forward_sharded(Xn2, p["W_up"], p["b_up"], p["W_down"], None, cfg["act"], t)
    Y_sh = reduce_scatter_seq(ml["P"], t) + _zeros_if_none(p["b_down"], X.shape[2]) + X1_sh
    return {"Xn1": Xn1, "m1": m1, "r1": r1, "attn": at, "X1": X1_sh, "Xn2": Xn2, "m2": m2,
            "r2": r2, "mlp": ml, "Y": Y_sh}


def layer_backward(G, X, p, cfg, t, fwd, sp=False):
    """Gradients of L = <Y, G> through :func:`layer_forward` (same layout as X)."""
    nh, dh = cfg["n_heads"], cfg["head_dim"]
    if not sp:
        mg = mlp_backward_sharded(G, fwd["Xn2"], p["W_up"], p["W_down"], fwd["mlp"], cfg["act"], t)
        dX1_ln, dg2, db2 = layernorm_backward(mg["dX"], fwd["X1"], p["ln2_g"], fwd["m2"], fwd["r2"])
        dX1 = G + dX1_ln
        ag = attn_backward_sharded(dX1, fwd["Xn1"], p["W_qkv"], p["W_o"], fwd["attn"], nh, dh,
                                   cfg["scale"], t)
        dX_ln, dg1, db1 = layernorm_backward(ag["dXn"], X, p["ln1_g"], fwd["m1"], fwd["r1"])
        dX = dX1 + dX_ln
    else:
        # ScatterSeq backward = all-gather of the shard grads; GatherSeq backward = reduce-scatter.
        Gf = all_gather_seq(G)
        mg = mlp_backward_sharded(Gf, fwd["Xn2"], p["W_up"], p["W_down"], fwd["mlp"], cfg["act"], t)
        dXn2_sh = reduce_scatter_seq(mg["dX_partials"], t)
        dX1_ln, _, _, dg2, db2 = sp_layernorm_backward(dXn2_sh, fwd["X1"], p["ln2_g"], fwd["m2"], fwd["r2"])
        dX1 = G + dX1_ln
        ag = attn_backward_sharded(all_gather_seq(dX1), fwd["Xn1"], p["W_qkv"], p["W_o"], fwd["attn"],
                                   nh, dh, cfg["scale"], t)
        dXn1_sh = reduce_scatter_seq(ag["dXn_partials"], t)
        dX_ln, _, _, dg1, db1 = sp_layernorm_backward(dXn1_sh, X, p["ln1_g"], fwd["m1"], fwd["r1"])
        dX = dX1 + dX_ln
    return {"dX": dX, "ln1_g": dg1, "ln1_b": db1, "ln2_g": dg2, "ln2_b": db2,
            "W_qkv": ag["dW_qkv"], "b_qkv": ag["db_qkv"], "W_o": ag["dW_o"], "b_o": ag["db_o"],
            "W_up": mg["dW_up"], "b_up": mg["db_up"], "W_down": mg["dW_down"], "b_down": mg["db_down"]}


def layer_forward_rows(X, p, cfg, t, rows):
    """:func:`layer_forward` (replicated LayerNorms) at the output rows `rows`
    only.  Attention needs every row's K and V, so the attention branch runs on
    all rows; LN2 and the MLP act row by row, so they run on `rows` alone.
    The sequence-parallel form gives the same rows (it only regroups them)."""
    nh, dh, eps = cfg["n_heads"], cfg["head_dim"], cfg["eps"]
    Xn1, _, _ = layernorm_forward(X, p["ln1_g"], p["ln1_b"], eps)
    at = attn_forward_sharded(Xn1, p["W_qkv"], p["b_qkv"], p["W_o"], p["b_o"], nh, dh, cfg["causal"],
                              cfg["scale"], t)
    X1 = X[rows] + at["Y"][rows]
    Xn2, _, _ = layernorm_forward(X1, p["ln2_g"], p["ln2_b"], eps)
    ml = mlp_forward_sharded(Xn2, p["W_up"], p["b_up"], p["W_down"], p["b_down"], cfg["act"], t)
    return {"X1": X1, "Y": X1 + ml["Y"]}


# ---------------------------------------------------------------------------
# Byte and FLOP accounting.
# ---------------------------------------------------------------------------

def expanded_tensor_bytes(tokens, expanded, elem_bytes):
    """Logical size of the sharded hidden tensor, tokens x expanded width."""
    return tokens * expanded * elem_bytes


def reduction_tensor_bytes(tokens, width, elem_bytes):
    """Logical size of the output-shaped tensor that the g all-reduce sums."""
    return tokens * width * elem_bytes


def allreduce_payload_bytes(batch, seq, hidden, elem_bytes):
    """b x s x h x bytes: the payload each TP all-reduce touches."""
    return batch * seq * hidden * elem_bytes


def mlp_fwd_bwd_flops(M, h, F):
    """Six GEMMs of 2*M*h*F each: Z, Y forward; dA, dX, dW_down, dW_up backward."""
    return 6 * 2 * M * h * F
