"""fp64 oracle, part 3: vocab-parallel embedding (test infrastructure only).

"Megatron-LM: Tensor Parallelism" (vanos001), section "Common Pitfalls",
item 5: the embedding lookup (token -> vector) is sharded by vocabulary.

Readings taken (the page states only the sharding):
* Shard i owns the contiguous vocabulary rows [i V/t, (i+1) V/t) of E (V, h).
* Forward: every shard receives all token ids (the f operator: identity);
  shard i returns E[id] for the ids it owns and zeros for the others; g sums
  the t partials (all-reduce forward, identity backward) -- exactly one partial
  is non-zero for every token.
* Backward: g backward hands dY to every shard unchanged; shard i adds
  dY[n] into its own row of dE for every token n whose id it owns (tokens in
  order); nothing is exchanged.
* The output (the LM head) would be the column-parallel GEMM against E^T with
  the same vocabulary split; the pages describe no loss, so none is built.
"""

from __future__ import annotations

import numpy as np

from .tp_oracle import shard_slice

__all__ = ["embedding_forward_unsplit", "embedding_forward_sharded", "embedding_backward_unsplit",
           "embedding_backward_sharded", "pack_vocab_rows"]


def embedding_forward_unsplit(ids, E):
    """Y[n] = E[ids[n]]."""
    return E[np.asarray(ids, dtype=np.int64)]


def embedding_forward_sharded(ids, E, t):
    """Per shard: its rows of E for the ids it owns, zero elsewhere; then g sums
    the t partials in shard order."""
    ids = np.asarray(ids, dtype=np.int64)
    V, h = E.shape
    partials = []
    for i in range(t):
        rows = shard_slice(V, t, i)
        E_i = E[rows]
        P = np.zeros((ids.size, h))
        mine = (ids >= rows.start) & (ids < rows.stop)
        P[mine] = E_i[ids[mine] - rows.start]
        partials.append(P)
    Y = np.zeros((ids.size, h))
    for i in range(t):
        Y = Y + partials[i]
    return {"Y": Y, "partials": partials}


def embedding_backward_unsplit(ids, dY, V):
    """dE[v] = sum of dY[n] over tokens n with ids[n] == v."""
    ids = np.asarray(ids, dtype=np.int64)
    dE = np.zeros((V, dY.shape[1]))
    np.add.at(dE, ids, dY)
    return dE


def embedding_backward_sharded(ids, dY, V, t):
    """Shard i: dE_i[v - i V/t] += dY[n] for the tokens it owns, in token order."""
    ids = np.asarray(ids, dtype=np.int64)
    out = []
    for i in range(t):
        rows = shard_slice(V, t, i)
        dE_i = np.zeros((rows.stop - rows.start, dY.shape[1]))
        for n in range(ids.size):
            if rows.start <= ids[n] < rows.stop:
                dE_i[ids[n] - rows.start] += dY[n]
        out.append(dE_i)
    return out


def pack_vocab_rows(E, t):
    """E (V, h) -> [t][V/t][h]: the shards' row blocks (already contiguous)."""
    V = E.shape[0]
    return np.stack([E[shard_slice(V, t, i)] for i in range(t)])
