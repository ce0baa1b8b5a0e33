"""Pins for the grouped-query and decode parts of the oracle.

Each check ties the oracle to something other than itself: the multi-head
oracle (already pinned by finite differences and closed forms) through the
exact identity "GQA = MHA with each KV head repeated over its group"; causal
prefill attention, of which a decode step is one row; brute-force finite
differences; closed forms (one key, equal scores); the numbers the roadmap page
prints for Llama-3-70B decode; and planted mistakes that the pins must catch.
"""

import json
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rand_gqa(rng, N, d, nh, nkv, hd, bias=True):
    W = rng.normal(scale=0.3, size=(d, (nh + 2 * nkv) * hd))
    b = rng.normal(scale=0.1, size=(nh + 2 * nkv) * hd) if bias else None
    Wo = rng.normal(scale=0.3, size=(nh * hd, d))
    bo = rng.normal(scale=0.1, size=d) if bias else None
    X = rng.normal(size=(N, d))
    return X, W, b, Wo, bo


def _fd(loss, arr, step=1e-6):
    flat = arr.reshape(-1)
    num = np.zeros(flat.size)
    for k in range(flat.size):
        old = flat[k]
        flat[k] = old + step; lp = loss()
        flat[k] = old - step; lm = loss()
        flat[k] = old
        num[k] = (lp - lm) / (2 * step)
    return num.reshape(arr.shape)


def _close(a, b, tol=1e-12):
    scale = max(np.abs(b).max(), 1e-30)
    assert np.abs(a - b).max() <= tol * scale, np.abs(a - b).max() / scale


# ---------------------------------------------------------------------------
# Layout.
# ---------------------------------------------------------------------------

def test_columns_reduce_to_multi_head_layout():
    for nh, hd, t in [(4, 2, 2), (8, 4, 4), (8, 3, 8)]:
        d = nh * hd
        for i in range(t):
            assert np.array_equal(O.gqa_qkv_shard_columns(nh, nh, hd, t, i),
                                  O.qkv_shard_columns(d, nh, hd, t, i))


def test_kv_heads_per_shard_and_replication():
    # n_kv >= t: disjoint groups covering all KV heads
    got = [list(O.gqa_shard_kv_heads(16, 8, 4, i)) for i in range(4)]
    assert got == [[0, 1], [2, 3], [4, 5], [6, 7]]
    # n_kv < t: each KV head on t/n_kv consecutive shards
    got = [list(O.gqa_shard_kv_heads(16, 2, 8, i)) for i in range(8)]
    assert got == [[0]] * 4 + [[1]] * 4
    # every query head of a shard reads one of the shard's KV heads
    for nh, nkv, t in [(16, 8, 4), (16, 2, 8), (8, 1, 4), (8, 8, 8)]:
        G = nh // nkv
        for i in range(t):
            kv = O.gqa_shard_kv_heads(nh, nkv, t, i)
            for j in range(i * nh // t, (i + 1) * nh // t):
                assert j // G in kv
    # the pages' cap: fewer KV heads than shards is only possible by replication
    with pytest.raises(AssertionError):
        O.gqa_shard_kv_heads(12, 3, 2, 0)      # 3 KV heads do not split over 2 shards


def test_pack_is_a_permutation_of_columns():
    rng = np.random.default_rng(1)
    nh, nkv, hd, t, d = 8, 2, 4, 4, 16
    W = rng.normal(size=(d, (nh + 2 * nkv) * hd))
    P = O.pack_qkv_gqa_weight(W, nh, nkv, hd, t)
    assert P.shape == (t, (nh // t + 2) * hd, d)
    for i in range(t):
        cols = O.gqa_qkv_shard_columns(nh, nkv, hd, t, i)
        for r, c in enumerate(cols):
            assert np.array_equal(P[i, r], W[:, c])
    # every Q column appears once; every K/V column t/n_kv times
    allc = np.concatenate([O.gqa_qkv_shard_columns(nh, nkv, hd, t, i) for i in range(t)])
    counts = np.bincount(allc, minlength=W.shape[1])
    assert (counts[:nh * hd] == 1).all() and (counts[nh * hd:] == t // nkv).all()


# ---------------------------------------------------------------------------
# Prefill GQA against the multi-head oracle.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("nh,nkv", [(4, 4), (4, 2), (4, 1), (6, 3)])
@pytest.mark.parametrize("causal", [True, False])
def test_gqa_equals_expanded_mha(nh, nkv, causal):
    rng = np.random.default_rng(2)
    hd, N = 3, 5
    d = nh * hd
    X, W, b, Wo, bo = _rand_gqa(rng, N, d, nh, nkv, hd)
    g = O.attn_gqa_forward_unsplit(X, W, b, Wo, bo, nh, nkv, hd, causal, 0.7)
    We, be = O.expand_gqa_to_mha(W, nh, nkv, hd), O.expand_gqa_to_mha(b, nh, nkv, hd)
    m = O.attn_forward_unsplit(X, We, be, Wo, bo, nh, hd, causal, 0.7)
    _close(g["Y"], m["Y"])
    # backward: Q and W_o gradients equal; a KV head's gradient is the sum of
    # its group's expanded copies
    Gy = rng.normal(size=g["Y"].shape)
    gb = O.attn_gqa_backward_unsplit(Gy, X, W, Wo, g, nh, nkv, hd, 0.7)
    mb = O.attn_backward_unsplit(Gy, X, We, Wo, m, nh, hd, 0.7)
    _close(gb["dXn"], mb["dXn"])
    _close(gb["dW_o"], mb["dW_o"])
    nq = nh * hd
    _close(gb["dW_qkv"][:, :nq], mb["dW_qkv"][:, :nq])
    G = nh // nkv
    for part in (1, 2):
        for gk in range(nkv):
            want = sum(mb["dW_qkv"][:, part * nq + j * hd: part * nq + (j + 1) * hd] for j in range(gk * G, (gk + 1) * G))
            got = gb["dW_qkv"][:, nq + (part - 1) * nkv * hd + gk * hd: nq + (part - 1) * nkv * hd + (gk + 1) * hd]
            _close(got, want)


@pytest.mark.parametrize("nh,nkv,t", [(8, 8, 4), (8, 2, 2), (8, 2, 4), (8, 2, 8), (8, 1, 4), (4, 4, 1)])
def test_gqa_sharded_equals_unsplit(nh, nkv, t):
    rng = np.random.default_rng(3)
    hd, N = 2, 4
    d = nh * hd
    X, W, b, Wo, bo = _rand_gqa(rng, N, d, nh, nkv, hd)
    U = O.attn_gqa_forward_unsplit(X, W, b, Wo, bo, nh, nkv, hd, True, 0.5)
    S = O.attn_gqa_forward_sharded(X, W, b, Wo, bo, nh, nkv, hd, True, 0.5, t)
    _close(S["Y"], U["Y"])
    Gy = rng.normal(size=U["Y"].shape)
    ub = O.attn_gqa_backward_unsplit(Gy, X, W, Wo, U, nh, nkv, hd, 0.5)
    sb = O.attn_gqa_backward_sharded(Gy, X, W, Wo, S, nh, nkv, hd, 0.5, t)
    for k in ("dXn", "dW_qkv", "db_qkv", "dW_o", "db_o"):
        _close(sb[k], ub[k])


def test_replicated_kv_gradient_needs_the_sum_over_copies():
    """With n_kv < t one copy's gradient is only a part of the shared weight's
    gradient; the copies sum to it."""
    rng = np.random.default_rng(4)
    nh, nkv, hd, t, N = 8, 2, 2, 8, 4
    X, W, b, Wo, bo = _rand_gqa(rng, N, nh * hd, nh, nkv, hd)
    U = O.attn_gqa_forward_unsplit(X, W, b, Wo, bo, nh, nkv, hd, True, 0.5)
    S = O.attn_gqa_forward_sharded(X, W, b, Wo, bo, nh, nkv, hd, True, 0.5, t)
    Gy = rng.normal(size=U["Y"].shape)
    ub = O.attn_gqa_backward_unsplit(Gy, X, W, Wo, U, nh, nkv, hd, 0.5)
    sb = O.attn_gqa_backward_sharded(Gy, X, W, Wo, S, nh, nkv, hd, 0.5, t)
    q_t = nh // t
    kcols = O.gqa_qkv_shard_columns(nh, nkv, hd, t, 0)[q_t * hd:(q_t + 1) * hd]
    one = sb["dWqkv_shard"][0][:, q_t * hd:(q_t + 1) * hd]
    assert np.abs(one - ub["dW_qkv"][:, kcols]).max() > 1e-3
    total = sum(sb["dWqkv_shard"][i][:, q_t * hd:(q_t + 1) * hd] for i in range(t // nkv))
    _close(total, ub["dW_qkv"][:, kcols])


def test_gqa_backward_finite_differences():
    rng = np.random.default_rng(5)
    nh, nkv, hd, N, t = 4, 2, 2, 3, 2
    d = nh * hd
    X, W, b, Wo, bo = _rand_gqa(rng, N, d, nh, nkv, hd)
    Gy = rng.normal(size=(N, d))

    def loss():
        return float((O.attn_gqa_forward_sharded(X, W, b, Wo, bo, nh, nkv, hd, True, 0.8, t)["Y"] * Gy).sum())

    S = O.attn_gqa_forward_sharded(X, W, b, Wo, bo, nh, nkv, hd, True, 0.8, t)
    g = O.attn_gqa_backward_sharded(Gy, X, W, Wo, S, nh, nkv, hd, 0.8, t)
    for name, arr, ana in [("X", X, g["dXn"]), ("W", W, g["dW_qkv"]), ("b", b, g["db_qkv"]),
                           ("Wo", Wo, g["dW_o"]), ("bo", bo, g["db_o"])]:
        num = _fd(loss, arr)
        err = np.abs(num - ana).max() / max(np.abs(num).max(), 1e-3)
        assert err <= 1e-6, (name, err)


def test_wrong_group_mapping_is_caught():
    """Planted mistake: query head j reading KV head j % n_kv instead of
    j // group gives a different output."""
    rng = np.random.default_rng(6)
    nh, nkv, hd, N = 4, 2, 2, 4
    X, W, b, Wo, bo = _rand_gqa(rng, N, nh * hd, nh, nkv, hd)
    good = O.attn_gqa_forward_unsplit(X, W, b, Wo, bo, nh, nkv, hd, True, 0.5)["Y"]
    nq = nh * hd
    idx = np.concatenate([np.arange((j % nkv) * hd, (j % nkv + 1) * hd) for j in range(nh)])
    k, v = W[:, nq:nq + nkv * hd], W[:, nq + nkv * hd:]
    kb, vb = b[nq:nq + nkv * hd], b[nq + nkv * hd:]
    We = np.concatenate([W[:, :nq], k[:, idx], v[:, idx]], axis=1)
    be = np.concatenate([b[:nq], kb[idx], vb[idx]])
    bad = O.attn_forward_unsplit(X, We, be, Wo, bo, nh, hd, True, 0.5)["Y"]
    assert np.abs(good - bad).max() > 1e-3


# ---------------------------------------------------------------------------
# Decode.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("nh,nkv", [(4, 4), (4, 2), (4, 1)])
def test_decode_steps_equal_causal_prefill_rows(nh, nkv):
    """Feeding the tokens one at a time through the cache reproduces causal
    attention over the whole sequence, row by row."""
    rng = np.random.default_rng(7)
    hd, N, L = 3, 6, 8
    d = nh * hd
    X, W, b, Wo, bo = _rand_gqa(rng, N, d, nh, nkv, hd)
    full = O.attn_gqa_forward_unsplit(X, W, b, Wo, bo, nh, nkv, hd, True, 0.6)["Y"]
    Kc = np.full((nkv, 1, L, hd), 7.0)      # stale contents beyond pos must not matter
    Vc = np.full((nkv, 1, L, hd), -3.0)
    for n in range(N):
        r = O.decode_attn_unsplit(X[n:n + 1], W, b, Wo, bo, Kc, Vc, [n], nh, nkv, hd, 0.6)
        _close(r["y"][0], full[n])
        Kc, Vc = r["K_cache"], r["V_cache"]


def test_decode_batch_is_independent_sequences():
    rng = np.random.default_rng(8)
    nh, nkv, hd, L, B = 4, 2, 2, 9, 3
    d = nh * hd
    X, W, b, Wo, bo = _rand_gqa(rng, B, d, nh, nkv, hd)
    Kc = rng.normal(size=(nkv, B, L, hd)); Vc = rng.normal(size=(nkv, B, L, hd))
    pos = [0, 5, 8]
    r = O.decode_attn_unsplit(X, W, b, Wo, bo, Kc, Vc, pos, nh, nkv, hd, 0.5)
    for bb in range(B):
        s = O.decode_attn_unsplit(X[bb:bb + 1], W, b, Wo, bo, Kc[:, bb:bb + 1], Vc[:, bb:bb + 1], [pos[bb]],
                                  nh, nkv, hd, 0.5)
        _close(r["y"][bb], s["y"][0])
    # only position pos[b] of each cache row changes, and holds x W_k + b_k
    nq = nh * hd
    for bb in range(B):
        for g in range(nkv):
            changed = np.where(np.abs(r["K_cache"][g, bb] - Kc[g, bb]).max(axis=1) > 0)[0]
            assert changed.tolist() == [pos[bb]]
            want = X[bb] @ W[:, nq + g * hd:nq + (g + 1) * hd] + b[nq + g * hd:nq + (g + 1) * hd]
            _close(r["K_cache"][g, bb, pos[bb]], want)


def test_decode_closed_forms():
    rng = np.random.default_rng(9)
    nh, nkv, hd, L = 4, 2, 3, 5
    d = nh * hd
    X, W, b, Wo, bo = _rand_gqa(rng, 1, d, nh, nkv, hd, bias=False)
    Kc = rng.normal(size=(nkv, 1, L, hd)); Vc = rng.normal(size=(nkv, 1, L, hd))
    # pos = 0: one key, softmax of one element -> O = the new value row
    r = O.decode_attn_unsplit(X, W, None, Wo, None, Kc, Vc, [0], nh, nkv, hd, 0.5)
    nq = nh * hd
    v = X[0] @ W[:, nq + nkv * hd:]
    for j in range(nh):
        g = j // (nh // nkv)
        _close(r["O"][0, j * hd:(j + 1) * hd], v[g * hd:(g + 1) * hd])
    # zero query weights: equal scores -> the mean of the visible value rows
    W0 = W.copy(); W0[:, :nq] = 0.0
    r = O.decode_attn_unsplit(X, W0, None, Wo, None, Kc, Vc, [3], nh, nkv, hd, 0.5)
    for j in range(nh):
        g = j // (nh // nkv)
        _close(r["O"][0, j * hd:(j + 1) * hd], r["V_cache"][g, 0, :4].mean(axis=0))


@pytest.mark.parametrize("nh,nkv,t", [(8, 8, 4), (8, 2, 2), (8, 2, 4), (8, 2, 8), (8, 1, 8), (4, 4, 1)])
def test_decode_sharded_equals_unsplit(nh, nkv, t):
    rng = np.random.default_rng(10)
    hd, L, B = 2, 7, 3
    d = nh * hd
    X, W, b, Wo, bo = _rand_gqa(rng, B, d, nh, nkv, hd)
    Kc = rng.normal(size=(nkv, B, L, hd)); Vc = rng.normal(size=(nkv, B, L, hd))
    pos = [2, 6, 0]
    U = O.decode_attn_unsplit(X, W, b, Wo, bo, Kc, Vc, pos, nh, nkv, hd, 0.5)
    Ks, Vs = O.shard_kv_cache(Kc, nh, nkv, t), O.shard_kv_cache(Vc, nh, nkv, t)
    S = O.decode_attn_sharded(X, W, b, Wo, bo, Ks, Vs, pos, nh, nkv, hd, 0.5, t)
    _close(S["y"], U["y"])
    # each shard's cache copy equals the unsplit cache's heads it holds;
    # replicated copies are identical
    _close(S["K_shards"], O.shard_kv_cache(U["K_cache"], nh, nkv, t))
    _close(S["V_shards"], O.shard_kv_cache(U["V_cache"], nh, nkv, t))


def test_decode_allreduce_accounting_matches_page():
    with open(os.path.join(GOLD, "page_payloads.json")) as f:
        L = json.load(f)["llama3_70b_decode"]
    a = O.decode_allreduce_accounting(L["batch"], L["hidden"], L["layers"], L["element_bytes"])
    assert a["payload_bytes"] == L["payload_bytes"]
    assert a["allreduces_per_layer"] == L["allreduces_per_layer_per_token"]
    assert a["allreduces_per_token"] == L["allreduces_per_token"]


def test_decode_bytes_count_every_copy():
    # Llama-3-70B-shaped attention at TP=4: Q 64 heads, 8 KV heads, 128 wide
    b4 = O.decode_attn_bytes(8192, 64, 8, 128, 4, [0])
    w = (64 + 16) * 128 * 8192 * 2 + 64 * 128 * 8192 * 2
    assert b4 == w + 2 * 8 * 1 * 128 * 2
    # TP=16 with 8 KV heads replicates each KV head twice: K/V weights and cache double
    b16 = O.decode_attn_bytes(8192, 64, 8, 128, 16, [9])
    w16 = (64 + 2 * 16) * 128 * 8192 * 2 + 64 * 128 * 8192 * 2
    assert b16 == w16 + 2 * 16 * 10 * 128 * 2
