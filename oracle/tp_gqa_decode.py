"""fp64 oracle, part 2: grouped-query attention under head sharding, and
decode attention over a head-sharded KV cache (test infrastructure only).

Sources:

* "02 — Tensor Parallelism" (project-fortress roadmap), section "The attention
  pairing": with GQA/MQA the heads are sharded by KV group, the pattern is
  otherwise the one of multi-head attention.  Section "The critical
  inference-time subtlety: KV cache also shards": each rank holds the KV heads
  of its own query heads, so the cache is split with them; with g KV groups the
  TP degree is capped at g.
* "Tensor and sequence parallelism" (ai-infra handbooks), exercise 1 and its
  answer: when the KV head count is smaller than the TP degree the KV heads are
  replicated, each sits on t/n_kv ranks, each rank still computes only its own
  query heads, and the KV weights and the KV cache exist in several copies.
* Same roadmap page, section "The count: two all-reduces per block per
  direction": one all-reduce per TP region, two per block per decode token,
  each of b x 1 x h elements; "Concrete numbers for Llama-3-70B" gives 16 KB and
  160 all-reduces per token.

Layout of the unsplit QKV weight: W_qkv is (d, (n_heads + 2 n_kv) * head_dim),
columns [Q head 0 .. n_heads-1 | K head 0 .. n_kv-1 | V head 0 .. n_kv-1], each
head head_dim wide.  Query head j reads KV head j // (n_heads / n_kv).

Readings taken where the pages are silent: the KV heads of a shard are the
groups of its query heads (contiguous query heads, contiguous groups); a
replicated KV head's weight gradient is the sum of its copies' gradients (the
same kind of sum the pages require for the LayerNorm weights shared across
sequence shards); a decode step appends the new token's key and value at
position pos[b] and attends to keys 0..pos[b] (the new token sees itself, as
row pos[b] of causal attention does).
"""

from __future__ import annotations

import numpy as np

from .tp_oracle import attention_head_backward, attention_head_forward, shard_slice, _zeros_if_none

__all__ = [
    "gqa_group", "gqa_shard_kv_heads", "gqa_qkv_shard_columns", "pack_qkv_gqa_weight",
    "pack_qkv_gqa_bias", "expand_gqa_to_mha",
    "attn_gqa_forward_unsplit", "attn_gqa_forward_sharded",
    "attn_gqa_backward_unsplit", "attn_gqa_backward_sharded",
    "shard_kv_cache", "decode_attn_unsplit", "decode_attn_sharded",
    "decode_allreduce_accounting", "decode_attn_bytes",
]


# ---------------------------------------------------------------------------
# Sharding by KV group.
# ---------------------------------------------------------------------------

def gqa_group(n_heads: int, n_kv: int) -> int:
    """Query heads per KV head."""
    assert n_heads % n_kv == 0
    return n_heads // n_kv


def gqa_shard_kv_heads(n_heads: int, n_kv: int, t: int, i: int) -> range:
    """Global KV heads that shard i holds.

    n_kv >= t: the n_kv/t groups of its query heads.  n_kv < t: the single KV
    head its query heads read, replicated on t/n_kv consecutive shards.
    """
    assert n_heads % t == 0 and n_heads % n_kv == 0
    if n_kv >= t:
        assert n_kv % t == 0
        s = shard_slice(n_kv, t, i)
        return range(s.start, s.stop)
    assert t % n_kv == 0
    j = (i * n_kv) // t
    return range(j, j + 1)


def gqa_qkv_shard_columns(n_heads: int, n_kv: int, head_dim: int, t: int, i: int) -> np.ndarray:
    """Columns of the unsplit W_qkv owned by shard i, in the order [its Q heads |
    its K heads | its V heads]."""
    qs = shard_slice(n_heads, t, i)
    kv = gqa_shard_kv_heads(n_heads, n_kv, t, i)
    q0, k0, v0 = 0, n_heads * head_dim, (n_heads + n_kv) * head_dim
    cols = []
    for j in range(qs.start, qs.stop):
        cols.extend(range(q0 + j * head_dim, q0 + (j + 1) * head_dim))
    for base in (k0, v0):
        for j in kv:
            cols.extend(range(base + j * head_dim, base + (j + 1) * head_dim))
    return np.asarray(cols, dtype=np.int64)


def pack_qkv_gqa_weight(Wqkv: np.ndarray, n_heads: int, n_kv: int, head_dim: int, t: int) -> np.ndarray:
    """W_qkv (d, (n_heads+2n_kv)*head_dim) -> [t][R][d], R = (n_heads/t + 2 kv_t)*head_dim:
    each shard's columns stored transposed (per-shard (out, in) weights)."""
    return np.stack([Wqkv[:, gqa_qkv_shard_columns(n_heads, n_kv, head_dim, t, i)].T for i in range(t)])


def pack_qkv_gqa_bias(b: np.ndarray, n_heads: int, n_kv: int, head_dim: int, t: int) -> np.ndarray:
    return np.stack([b[gqa_qkv_shard_columns(n_heads, n_kv, head_dim, t, i)] for i in range(t)])


def expand_gqa_to_mha(W: np.ndarray, n_heads: int, n_kv: int, head_dim: int) -> np.ndarray:
    """Repeat each KV head's columns for every query head of its group: the
    multi-head weight (d, 3 n_heads head_dim) that computes the same attention.
    Works on weights (2-D) and biases (1-D)."""
    G = gqa_group(n_heads, n_kv)
    nq = n_heads * head_dim
    q = W[..., :nq]
    k = W[..., nq:nq + n_kv * head_dim]
    v = W[..., nq + n_kv * head_dim:]
    idx = np.concatenate([np.arange((j // G) * head_dim, (j // G + 1) * head_dim) for j in range(n_heads)])
    return np.concatenate([q, k[..., idx], v[..., idx]], axis=-1)


def _q_cols(j, hd):
    return slice(j * hd, (j + 1) * hd)


# ---------------------------------------------------------------------------
# Grouped-query attention (prefill), unsplit and sharded.
# ---------------------------------------------------------------------------

def attn_gqa_forward_unsplit(Xn, W_qkv, b_qkv, W_o, b_o, n_heads, n_kv, head_dim, causal, scale):
    N = Xn.shape[0]
    G = gqa_group(n_heads, n_kv)
    nq, nk = n_heads * head_dim, n_kv * head_dim
    QKV = Xn @ W_qkv + _zeros_if_none(b_qkv, nq + 2 * nk)
    Q, K, V = QKV[:, :nq], QKV[:, nq:nq + nk], QKV[:, nq + nk:]
    O = np.zeros((N, nq))
    Ps, lses = [], []
    for j in range(n_heads):
        g = j // G
        o, p, lse = attention_head_forward(Q[:, _q_cols(j, head_dim)], K[:, _q_cols(g, head_dim)],
                                           V[:, _q_cols(g, head_dim)], causal, scale)
        O[:, _q_cols(j, head_dim)] = o
        Ps.append(p); lses.append(lse)
    Y = O @ W_o + _zeros_if_none(b_o, W_o.shape[1])
    return {"QKV": QKV, "O": O, "P": Ps, "lse": np.stack(lses), "Y": Y}


def attn_gqa_forward_sharded(Xn, W_qkv, b_qkv, W_o, b_o, n_heads, n_kv, head_dim, causal, scale, t):
    """Shard i: its query heads and the KV heads they read (replicated copies
    when n_kv < t), attention on its query heads, its rows of W_o; g sums the
    t partials, output bias once."""
    N = Xn.shape[0]
    G = gqa_group(n_heads, n_kv)
    q_t = n_heads // t
    b_qkv = _zeros_if_none(b_qkv, W_qkv.shape[1])
    QKVs, Os, Ps, partials = [], [], [], []
    for i in range(t):
        cols = gqa_qkv_shard_columns(n_heads, n_kv, head_dim, t, i)
        kv = gqa_shard_kv_heads(n_heads, n_kv, t, i)
        kv_t = len(kv)
        QKV_i = Xn @ W_qkv[:, cols] + b_qkv[cols]
        Qi = QKV_i[:, :q_t * head_dim]
        Ki = QKV_i[:, q_t * head_dim:(q_t + kv_t) * head_dim]
        Vi = QKV_i[:, (q_t + kv_t) * head_dim:]
        O_i = np.zeros((N, q_t * head_dim))
        for jj in range(q_t):
            jl = (i * q_t + jj) // G - kv.start          # local KV head of this query head
            o, p, _ = attention_head_forward(Qi[:, _q_cols(jj, head_dim)], Ki[:, _q_cols(jl, head_dim)],
                                             Vi[:, _q_cols(jl, head_dim)], causal, scale)
            O_i[:, _q_cols(jj, head_dim)] = o
            Ps.append(p)
        partials.append(O_i @ W_o[shard_slice(n_heads * head_dim, t, i), :])
        QKVs.append(QKV_i); Os.append(O_i)
    Y = np.zeros((N, W_o.shape[1]))
    for i in range(t):
        Y = Y + partials[i]
    Y = Y + _zeros_if_none(b_o, W_o.shape[1])
    return {"QKV": QKVs, "O": Os, "P": Ps, "partials": partials, "Y": Y}


def attn_gqa_backward_unsplit(Gy, Xn, W_qkv, W_o, fwd, n_heads, n_kv, head_dim, scale):
    """Gradients of L = <Y, Gy>.  A KV head's dK/dV is the sum over the query
    heads of its group."""
    G = gqa_group(n_heads, n_kv)
    nq, nk = n_heads * head_dim, n_kv * head_dim
    QKV = fwd["QKV"]
    Q, K, V = QKV[:, :nq], QKV[:, nq:nq + nk], QKV[:, nq + nk:]
    dO = Gy @ W_o.T
    dQKV = np.zeros_like(QKV)
    for j in range(n_heads):
        g = j // G
        dq, dk, dv = attention_head_backward(dO[:, _q_cols(j, head_dim)], Q[:, _q_cols(j, head_dim)],
                                             K[:, _q_cols(g, head_dim)], V[:, _q_cols(g, head_dim)],
                                             fwd["P"][j], scale)
        dQKV[:, _q_cols(j, head_dim)] = dq
        dQKV[:, nq + g * head_dim:nq + (g + 1) * head_dim] += dk
        dQKV[:, nq + nk + g * head_dim:nq + nk + (g + 1) * head_dim] += dv
    return {"dXn": dQKV @ W_qkv.T, "dW_qkv": Xn.T @ dQKV, "db_qkv": dQKV.sum(axis=0),
            "dW_o": fwd["O"].T @ Gy, "db_o": Gy.sum(axis=0), "dQKV": dQKV}


def attn_gqa_backward_sharded(Gy, Xn, W_qkv, W_o, fwd, n_heads, n_kv, head_dim, scale, t):
    """Per shard: dO_i = Gy W_o[rows_i]^T, head-local softmax backward, dK/dV
    summed over the shard's own query heads of each local KV head, the shard's
    weight gradient for its copy of the columns; f backward sums dXn.

    Returns the per-shard copy gradients ``dWqkv_shard`` ([t][d][R]) and the
    unsplit gradient ``dW_qkv`` in which the copies of a replicated KV head are
    summed in shard order.
    """
    G = gqa_group(n_heads, n_kv)
    q_t = n_heads // t
    dW_qkv = np.zeros_like(W_qkv)
    db_qkv = np.zeros(W_qkv.shape[1])
    dW_o = np.zeros_like(W_o)
    dXn = np.zeros_like(Xn)
    copies, bcopies, dQKVs = [], [], []
    for i in range(t):
        cols = gqa_qkv_shard_columns(n_heads, n_kv, head_dim, t, i)
        kv = gqa_shard_kv_heads(n_heads, n_kv, t, i)
        kv_t = len(kv)
        rows = shard_slice(n_heads * head_dim, t, i)
        QKV_i = fwd["QKV"][i]
        qo, ko, vo = 0, q_t * head_dim, (q_t + kv_t) * head_dim
        dO_i = Gy @ W_o[rows, :].T
        dW_o[rows, :] = fwd["O"][i].T @ Gy
        dQKV_i = np.zeros_like(QKV_i)
        for jj in range(q_t):
            jl = (i * q_t + jj) // G - kv.start
            kc = slice(ko + jl * head_dim, ko + (jl + 1) * head_dim)
            vc = slice(vo + jl * head_dim, vo + (jl + 1) * head_dim)
            qc = slice(qo + jj * head_dim, qo + (jj + 1) * head_dim)
            dq, dk, dv = attention_head_backward(dO_i[:, _q_cols(jj, head_dim)], QKV_i[:, qc], QKV_i[:, kc],
                                                 QKV_i[:, vc], fwd["P"][i * q_t + jj], scale)
            dQKV_i[:, qc] = dq
            dQKV_i[:, kc] += dk
            dQKV_i[:, vc] += dv
        dW_i = Xn.T @ dQKV_i
        db_i = dQKV_i.sum(axis=0)
        copies.append(dW_i); bcopies.append(db_i); dQKVs.append(dQKV_i)
        dW_qkv[:, cols] += dW_i          # replicated columns: copies summed in shard order
        db_qkv[cols] += db_i
        dXn = dXn + dQKV_i @ W_qkv[:, cols].T
    return {"dXn": dXn, "dW_qkv": dW_qkv, "db_qkv": db_qkv, "dW_o": dW_o, "db_o": Gy.sum(axis=0),
            "dWqkv_shard": copies, "dbqkv_shard": bcopies, "dQKV": dQKVs}


# ---------------------------------------------------------------------------
# Decode: one new token per sequence against a KV cache.
# ---------------------------------------------------------------------------

def shard_kv_cache(cache: np.ndarray, n_heads: int, n_kv: int, t: int) -> np.ndarray:
    """Unsplit cache [n_kv][B][L][hd] -> per-shard copies [t][kv_t][B][L][hd]."""
    return np.stack([cache[list(gqa_shard_kv_heads(n_heads, n_kv, t, i))] for i in range(t)])


def _decode_head(q, Kc, Vc, n_keys, scale):
    """One query row against keys 0..n_keys-1 of one cached head: the last row
    of causal attention over those keys."""
    s = scale * (Kc[:n_keys] @ q)
    m = s.max()
    e = np.exp(s - m)
    p = e / e.sum()
    return p @ Vc[:n_keys]


def decode_attn_unsplit(x, W_qkv, b_qkv, W_o, b_o, K_cache, V_cache, pos, n_heads, n_kv, head_dim, scale):
    """x [B][d]; caches [n_kv][B][L][hd]; pos [B].  Returns y [B][d'], the
    caches with the new keys/values written at pos[b], and q/O."""
    B = x.shape[0]
    G = gqa_group(n_heads, n_kv)
    nq, nk = n_heads * head_dim, n_kv * head_dim
    qkv = x @ W_qkv + _zeros_if_none(b_qkv, nq + 2 * nk)
    Kc, Vc = K_cache.copy(), V_cache.copy()
    O = np.zeros((B, nq))
    for b in range(B):
        p = int(pos[b])
        for g in range(n_kv):
            Kc[g, b, p] = qkv[b, nq + g * head_dim:nq + (g + 1) * head_dim]
            Vc[g, b, p] = qkv[b, nq + nk + g * head_dim:nq + nk + (g + 1) * head_dim]
        for j in range(n_heads):
            O[b, _q_cols(j, head_dim)] = _decode_head(qkv[b, _q_cols(j, head_dim)], Kc[j // G, b], Vc[j // G, b],
                                                       p + 1, scale)
    y = O @ W_o + _zeros_if_none(b_o, W_o.shape[1])
    return {"y": y, "K_cache": Kc, "V_cache": Vc, "qkv": qkv, "O": O}


def decode_attn_sharded(x, W_qkv, b_qkv, W_o, b_o, K_shards, V_shards, pos, n_heads, n_kv, head_dim, scale, t):
    """Per-shard caches [t][kv_t][B][L][hd].  Shard i projects its own Q/K/V
    columns, writes its KV heads' new entries into its own cache copy, attends
    with its query heads and forms its partial O_i W_o[rows_i]; g sums the t
    partials (one all-reduce of B x d' elements) and adds the output bias once."""
    B = x.shape[0]
    G = gqa_group(n_heads, n_kv)
    q_t = n_heads // t
    b_qkv = _zeros_if_none(b_qkv, W_qkv.shape[1])
    Ks, Vs = K_shards.copy(), V_shards.copy()
    partials, Os = [], []
    for i in range(t):
        cols = gqa_qkv_shard_columns(n_heads, n_kv, head_dim, t, i)
        kv = gqa_shard_kv_heads(n_heads, n_kv, t, i)
        kv_t = len(kv)
        qkv_i = x @ W_qkv[:, cols] + b_qkv[cols]
        ko, vo = q_t * head_dim, (q_t + kv_t) * head_dim
        O_i = np.zeros((B, q_t * head_dim))
        for b in range(B):
            p = int(pos[b])
            for jl in range(kv_t):
                Ks[i, jl, b, p] = qkv_i[b, ko + jl * head_dim:ko + (jl + 1) * head_dim]
                Vs[i, jl, b, p] = qkv_i[b, vo + jl * head_dim:vo + (jl + 1) * head_dim]
            for jj in range(q_t):
                jl = (i * q_t + jj) // G - kv.start
                O_i[b, _q_cols(jj, head_dim)] = _decode_head(qkv_i[b, _q_cols(jj, head_dim)], Ks[i, jl, b],
                                                              Vs[i, jl, b], p + 1, scale)
        partials.append(O_i @ W_o[shard_slice(n_heads * head_dim, t, i), :])
        Os.append(O_i)
    y = np.zeros((B, W_o.shape[1]))
    for i in range(t):
        y = y + partials[i]
    y = y + _zeros_if_none(b_o, W_o.shape[1])
    return {"y": y, "K_shards": Ks, "V_shards": Vs, "O": Os, "partials": partials}


# ---------------------------------------------------------------------------
# Accounting.
# ---------------------------------------------------------------------------

def decode_allreduce_accounting(batch, hidden, layers, elem_bytes):
    """All-reduces of a TP decode step: one per TP region (attention, MLP), so
    two per layer per token, each over batch x 1 x hidden elements."""
    payload = batch * 1 * hidden * elem_bytes
    per_layer = 2
    return {"payload_bytes": payload, "allreduces_per_layer": per_layer,
            "allreduces_per_token": per_layer * layers, "bytes_per_token": per_layer * layers * payload}


def decode_attn_bytes(d, n_heads, n_kv, head_dim, t, lengths, w_bytes=2, kv_bytes=2):
    """Algorithmic HBM bytes of one TP decode-attention step: the packed QKV
    weights of all shards (replicated KV columns counted once per copy), the
    cached keys and values each shard reads (lengths[b] + 1 positions each,
    per copy) and W_o.  Activations (B x d) are negligible and not counted."""
    kv_t = len(gqa_shard_kv_heads(n_heads, n_kv, t, 0))
    rows = t * (n_heads // t + 2 * kv_t) * head_dim
    w = rows * d * w_bytes + n_heads * head_dim * d * w_bytes
    kv = 0
    for L in lengths:
        kv += 2 * t * kv_t * (int(L) + 1) * head_dim * kv_bytes
    return w + kv
