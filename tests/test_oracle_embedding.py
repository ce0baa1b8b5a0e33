"""Pins for the vocab-parallel embedding oracle: the one-hot matrix product
(an independent formulation of a lookup), sharded = unsplit for every t, the
gradient by finite differences and by the transposed one-hot product, shard
boundaries and repeated ids, and a planted mistake."""

import numpy as np
import pytest

import oracle as O


def _onehot(ids, V):
    M = np.zeros((len(ids), V))
    M[np.arange(len(ids)), ids] = 1.0
    return M


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_lookup_equals_onehot_product_and_shards_agree(t):
    rng = np.random.default_rng(t)
    V, h, N = 64, 5, 40
    E = rng.normal(size=(V, h))
    ids = rng.integers(0, V, size=N)
    ids[:4] = [0, V - 1, V // t - 1 if t > 1 else 1, V // t if t > 1 else 2]  # shard boundaries
    ids[4:8] = 7  # repeats
    U = O.embedding_forward_unsplit(ids, E)
    assert np.array_equal(U, _onehot(ids, V) @ E)
    S = O.embedding_forward_sharded(ids, E, t)
    assert np.array_equal(S["Y"], U)
    # exactly one shard contributes each token
    nz = sum((np.abs(P).sum(axis=1) > 0).astype(int) for P in S["partials"])
    assert (nz == 1).all()


@pytest.mark.parametrize("t", [1, 2, 4])
def test_gradient_is_transposed_onehot_and_matches_shards(t):
    rng = np.random.default_rng(10 + t)
    V, h, N = 32, 3, 25
    ids = rng.integers(0, V, size=N)
    ids[:5] = 3
    dY = rng.normal(size=(N, h))
    dE = O.embedding_backward_unsplit(ids, dY, V)
    assert np.allclose(dE, _onehot(ids, V).T @ dY, rtol=0, atol=1e-12)
    parts = O.embedding_backward_sharded(ids, dY, V, t)
    assert np.allclose(np.concatenate(parts), dE, rtol=0, atol=1e-12)


def test_gradient_finite_differences():
    rng = np.random.default_rng(3)
    V, h, N, t = 8, 2, 6, 2
    E = rng.normal(size=(V, h))
    ids = np.array([1, 5, 1, 7, 0, 4])
    G = rng.normal(size=(N, h))
    ana = np.concatenate(O.embedding_backward_sharded(ids, G, V, t))
    num = np.zeros_like(E)
    for v in range(V):
        for j in range(h):
            old = E[v, j]
            E[v, j] = old + 1e-6; lp = (O.embedding_forward_sharded(ids, E, t)["Y"] * G).sum()
            E[v, j] = old - 1e-6; lm = (O.embedding_forward_sharded(ids, E, t)["Y"] * G).sum()
            E[v, j] = old
            num[v, j] = (lp - lm) / 2e-6
    assert np.abs(num - ana).max() <= 1e-6 * max(np.abs(num).max(), 1.0)


def test_planted_mistakes_are_caught():
    """Every shard looking up every token (no ownership mask) makes g count each
    embedding t times; a shard reading its slice at the global id reads another
    token's row."""
    rng = np.random.default_rng(4)
    V, h, t = 16, 3, 4
    E = rng.normal(size=(V, h))
    ids = np.array([5, 9, 14, 2])
    good = O.embedding_forward_sharded(ids, E, t)["Y"]
    no_mask = sum(E[ids] for _ in range(t))
    assert np.abs(good - no_mask).max() > 1e-3
    blk = V // t
    no_offset = np.stack([E[(v // blk) * blk:(v // blk + 1) * blk][v % blk] if v < blk else
                          E[(v // blk) * blk + (v % blk + 1) % blk] for v in ids])
    assert np.abs(good - no_offset).max() > 1e-3


def test_pack_is_row_blocks():
    E = np.arange(24.0).reshape(8, 3)
    P = O.pack_vocab_rows(E, 4)
    assert P.shape == (4, 2, 3) and np.array_equal(P.reshape(8, 3), E)
