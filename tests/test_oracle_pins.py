"""Pins for the fp64 oracle: values the pages print, closed forms, invariants,
negative cases the pages describe, and brute-force finite differences.

None of these compare the oracle with a retyped copy of itself: each check is
either a number printed on a page, an identity the mathematics fixes, or an
independent computation (finite differences, torch autograd in float64 as the
pages' own checks use it, math.erf).
"""

import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Worked example: "Tensor Parallelism's Communication Boundary".
# ---------------------------------------------------------------------------

def test_worked_example_exact_values():
    g = _gold("p3_worked_example.json")
    x = np.array([g["x"]], dtype=np.float64)
    w1 = np.array(g["w1"], dtype=np.float64)
    w2 = np.array(g["w2"], dtype=np.float64)
    un = O.mlp_forward_unsplit(x, w1, None, w2, None, "relu")
    assert un["Z"][0].tolist() == g["pre_activation"]
    assert un["Y"][0].tolist() == g["dense"]
    sh = O.mlp_forward_sharded(x, w1, None, w2, None, "relu", t=2)
    # the two workers own columns (0, 1) and (2, 3)
    assert [list(range(O.shard_slice(4, 2, i).start, O.shard_slice(4, 2, i).stop)) for i in range(2)] \
        == g["worker_columns"]
    assert [a[0].tolist() for a in sh["A"]] == g["local_hidden"]
    assert [p[0].tolist() for p in sh["P"]] == g["partials"]
    assert sh["Y"][0].tolist() == g["split"] == g["dense"]


def test_worked_example_bytes():
    b = _gold("p3_worked_example.json")["bytes"]
    e = O.expanded_tensor_bytes(b["tokens"], b["expanded"], b["element_bytes"])
    r = O.reduction_tensor_bytes(b["tokens"], b["width"], b["element_bytes"])
    assert e == b["expanded_tensor_bytes"]
    assert r == b["output_reduction_tensor_bytes"]
    assert e == b["ratio"] * r


def test_page_payload_numbers():
    g = _gold("page_payloads.json")
    L = g["llama3_70b_decode"]
    assert O.allreduce_payload_bytes(L["batch"], L["seq"], L["hidden"], L["element_bytes"]) == L["payload_bytes"]
    assert L["allreduces_per_layer_per_token"] * L["layers"] == L["allreduces_per_token"]
    G = g["gpt3_scale"]
    p = O.allreduce_payload_bytes(1, G["tokens"], G["hidden"], G["element_bytes"])
    assert abs(p - G["payload_bytes_approx"]) <= G["rel_tol"] * G["payload_bytes_approx"]
    assert 2 * G["layers"] == G["allreduces_per_forward"]


def test_rowfirst_split_is_wrong():
    g = _gold("p3_worked_example.json")
    c = g["counterexample"]
    relu = lambda v: O.act("relu", np.array([float(v)]))[0]
    assert relu(c["a"] + c["b"]) == c["relu_of_sum"]
    assert relu(c["a"]) + relu(c["b"]) == c["sum_of_relu"]
    x = np.array([g["x"]], dtype=np.float64)
    w1 = np.array(g["w1"], dtype=np.float64)
    w2 = np.array(g["w2"], dtype=np.float64)
    wrong = O.mlp_forward_rowfirst_split(x, w1, None, w2, None, "relu", t=2)
    assert wrong[0].tolist() != g["dense"]
    # with a linear activation the row-first split is harmless: the failure is the nonlinearity
    lin_ok = O.mlp_forward_rowfirst_split(x, w1, None, w2, None, "identity", t=2)
    assert np.allclose(lin_ok, O.mlp_forward_unsplit(x, w1, None, w2, None, "identity")["Y"], atol=0)


@pytest.mark.parametrize("t", [2, 4, 8])
def test_bias_added_once(t):
    rng = np.random.default_rng(t)
    X, Wu, bu, Wd, bd = rng.normal(size=(5, 8)), rng.normal(size=(8, 16)), rng.normal(size=16), \
        rng.normal(size=(16, 8)), rng.normal(size=8)
    good = O.mlp_forward_sharded(X, Wu, bu, Wd, bd, "gelu_tanh", t)["Y"]
    bad = O.mlp_forward_bias_every_shard(X, Wu, bu, Wd, bd, "gelu_tanh", t)
    assert np.allclose(bad - good, (t - 1) * bd[None, :], rtol=0, atol=1e-12)
    assert np.allclose(good, O.mlp_forward_unsplit(X, Wu, bu, Wd, bd, "gelu_tanh")["Y"], rtol=0, atol=1e-12)


@pytest.mark.parametrize("t", [2, 4])
def test_fg_swapped_is_wrong(t):
    rng = np.random.default_rng(7)
    X, Wu, bu, Wd, bd, G = rng.normal(size=(4, 8)), rng.normal(size=(8, 16)), rng.normal(size=16), \
        rng.normal(size=(16, 8)), rng.normal(size=8), rng.normal(size=(4, 8))
    ref = O.mlp_forward_unsplit(X, Wu, bu, Wd, bd, "gelu_tanh")
    refb = O.mlp_backward_unsplit(G, X, Wu, Wd, ref["Z"], ref["A"], "gelu_tanh")
    out0, dX0 = O.mlp_fg_swapped(X, Wu, bu, Wd, bd, "gelu_tanh", t, G)
    assert np.abs(out0 - ref["Y"]).max() > 1e-3
    assert np.abs(dX0 - refb["dX"]).max() > 1e-3
    # identity activation, no biases: input inflated t times and only shard 0's partial
    # survives, so rank 0's output is exactly t * P_0(X).
    out_lin, _ = O.mlp_fg_swapped(X, Wu, None, Wd, None, "identity", t, G)
    P0 = O.mlp_forward_sharded(X, Wu, None, Wd, None, "identity", t)["P"][0]
    assert np.allclose(out_lin, t * P0, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# Sharded == unsplit for every t; t = 1 is literally the unsplit block.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("act", O.ACTIVATIONS)
@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_sharded_equals_unsplit(act, t):
    rng = np.random.default_rng(100 + t)
    M, h, F = 7, 24, 64
    X, Wu, bu, Wd, bd, G = rng.normal(size=(M, h)), rng.normal(size=(h, F)) * 0.3, rng.normal(size=F), \
        rng.normal(size=(F, h)) * 0.3, rng.normal(size=h), rng.normal(size=(M, h))
    U = O.mlp_forward_unsplit(X, Wu, bu, Wd, bd, act)
    S = O.mlp_forward_sharded(X, Wu, bu, Wd, bd, act, t)
    tol = 1e-12 * np.abs(U["Y"]).max()
    assert np.abs(S["Y"] - U["Y"]).max() <= tol
    assert np.array_equal(np.concatenate(S["A"], axis=1), U["A"]) or \
        np.abs(np.concatenate(S["A"], axis=1) - U["A"]).max() <= 1e-12 * np.abs(U["A"]).max()
    Ub = O.mlp_backward_unsplit(G, X, Wu, Wd, U["Z"], U["A"], act)
    Sb = O.mlp_backward_sharded(G, X, Wu, Wd, S, act, t)
    for k in ("dX", "dW_up", "dW_down", "db_up", "db_down"):
        assert np.abs(Sb[k] - Ub[k]).max() <= 1e-12 * max(np.abs(Ub[k]).max(), 1.0), k
    # f backward: dX is the sum of the per-shard partials
    assert np.allclose(sum(Sb["dX_partials"]), Sb["dX"], rtol=0, atol=1e-12)
    if t == 1:
        assert np.array_equal(S["Y"], U["Y"])


# ---------------------------------------------------------------------------
# Brute-force central finite differences (fp64) on tiny shapes.
# ---------------------------------------------------------------------------

def _fd_check(loss, params, grads, step=1e-6, rtol=1e-6):
    for name, arr in params.items():
        g = grads[name]
        flat = arr.reshape(-1)
        num = np.zeros(flat.size)
        for k in range(flat.size):
            old = flat[k]
            flat[k] = old + step
            lp = loss()
            flat[k] = old - step
            lm = loss()
            flat[k] = old
            num[k] = (lp - lm) / (2 * step)
        ana = g.reshape(-1)
        scale = max(np.abs(num).max(), 1e-3)
        err = np.abs(num - ana).max() / scale
        assert err <= rtol, (name, err)


@pytest.mark.parametrize("act", O.ACTIVATIONS)
@pytest.mark.parametrize("t", [1, 2, 4])
def test_mlp_backward_finite_differences(act, t):
    rng = np.random.default_rng(11)
    M, h, F = 3, 4, 8
    X = rng.normal(size=(M, h)); Wu = rng.normal(size=(h, F)); bu = rng.normal(size=F)
    Wd = rng.normal(size=(F, h)); bd = rng.normal(size=h); G = rng.normal(size=(M, h))
    if act == "relu":
        assert np.abs(X @ Wu + bu).min() > 1e-3   # stay away from the kink
    p = {"X": X, "W_up": Wu, "b_up": bu, "W_down": Wd, "b_down": bd}

    def loss():
        return float((O.mlp_forward_sharded(X, Wu, bu, Wd, bd, act, t)["Y"] * G).sum())

    f = O.mlp_forward_sharded(X, Wu, bu, Wd, bd, act, t)
    b = O.mlp_backward_sharded(G, X, Wu, Wd, f, act, t)
    _fd_check(loss, p, {"X": b["dX"], "W_up": b["dW_up"], "b_up": b["db_up"],
                        "W_down": b["dW_down"], "b_down": b["db_down"]})


@pytest.mark.parametrize("t", [1, 2])
def test_swiglu_finite_differences(t):
    rng = np.random.default_rng(12)
    M, h, F = 3, 4, 8
    X = rng.normal(size=(M, h)); Wg = rng.normal(size=(h, F)); Wu = rng.normal(size=(h, F))
    Wd = rng.normal(size=(F, h)); G = rng.normal(size=(M, h))
    loss = lambda: float((O.swiglu_forward_sharded(X, Wg, Wu, Wd, t)["Y"] * G).sum())
    f = O.swiglu_forward_sharded(X, Wg, Wu, Wd, t)
    assert np.abs(f["Y"] - O.swiglu_forward_unsplit(X, Wg, Wu, Wd)["Y"]).max() < 1e-12
    b = O.swiglu_backward_sharded(G, X, Wg, Wu, Wd, f, t)
    _fd_check(loss, {"X": X, "W_gate": Wg, "W_up": Wu, "W_down": Wd},
              {"X": b["dX"], "W_gate": b["dW_gate"], "W_up": b["dW_up"], "W_down": b["dW_down"]})


# ---------------------------------------------------------------------------
# Activation closed forms.
# ---------------------------------------------------------------------------

def test_gelu_closed_forms():
    z = np.linspace(-6, 6, 241)
    for name in ("gelu_tanh", "gelu_erf"):
        # phi(z) - phi(-z) = z for any GeLU built as z * (symmetric CDF)
        assert np.allclose(O.act(name, z) - O.act(name, -z), z, atol=1e-14)
        assert O.act(name, np.array([0.0]))[0] == 0.0
        assert abs(O.act_grad(name, np.array([0.0]))[0] - 0.5) < 1e-15
        h = 1e-6
        num = (O.act(name, z + h) - O.act(name, z - h)) / (2 * h)
        assert np.abs(num - O.act_grad(name, z)).max() < 1e-8
    erf_ref = np.array([0.5 * v * (1 + math.erf(v / math.sqrt(2))) for v in z])
    assert np.abs(O.act("gelu_erf", z) - erf_ref).max() < 1e-15
    # the tanh form approximates the erf form to a few 1e-4 (Hendrycks & Gimpel)
    assert np.abs(O.act("gelu_tanh", z) - O.act("gelu_erf", z)).max() < 1e-3
    num = (O.silu(z + 1e-6) - O.silu(z - 1e-6)) / 2e-6
    assert np.abs(num - O.silu_grad(z)).max() < 1e-8


def test_silu_pins():
    """silu(z) = z * sigmoid(z), the gate of SwiGLU ("02 — Tensor Parallelism", "The
    core observation": the MLP's FLOPs "times 2 for SwiGLU").  Pinned by identities a
    wrong formula breaks: silu(z) - silu(-z) = z (sigmoid(z) + sigmoid(-z) = 1),
    silu(0) = 0, silu'(0) = 1/2, and the asymptotes silu(z) -> z, silu(-z) -> 0 with
    the exponentially small gap z e^{-z}."""
    z = np.linspace(-12, 12, 481)
    assert np.abs((O.silu(z) - O.silu(-z)) - z).max() < 1e-14
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert abs(O.silu_grad(np.array([0.0]))[0] - 0.5) < 1e-16
    big = np.array([30.0, 40.0])
    gap = big * np.exp(-big)                 # z - silu(z) = z e^{-z} / (1 + e^{-z})
    # above: silu(z) = z - z e^{-z} / (1 + e^{-z}), equal to z within rounding of z
    assert np.abs(O.silu(big) - (big - gap / (1 + np.exp(-big)))).max() <= 4 * np.spacing(big).max()
    # below: silu(-z) = -z e^{-z} / (1 + e^{-z}), a tiny value computed without cancellation
    assert np.allclose(-O.silu(-big), gap / (1 + np.exp(-big)), rtol=1e-12, atol=0)
    # the derivative tends to 1 above and 0 below
    assert abs(O.silu_grad(np.array([40.0]))[0] - 1.0) < 1e-15
    assert abs(O.silu_grad(np.array([-40.0]))[0]) < 1e-15


def _torch_f64(fn, z):
    import torch
    return fn(torch.from_numpy(np.asarray(z, dtype=np.float64))).numpy()


def test_activations_match_an_independent_library_in_fp64():
    """The oracle's activations against torch's own float64 implementations (a
    separate code base): SiLU, GeLU with the tanh approximation (this pins the cubic
    coefficient 0.044715 and sqrt(2/pi): a coefficient off by 1e-4 moves the value by
    ~1e-5 at |z| ~ 2, far above 1e-14) and exact GeLU; and their derivatives against
    torch autograd in float64."""
    import torch
    import torch.nn.functional as Fn
    z = np.concatenate([np.linspace(-10, 10, 2001), [-1e-8, 1e-8, 0.0, 3.7, -2.3]])
    assert np.abs(O.silu(z) - _torch_f64(Fn.silu, z)).max() <= 1e-14 * max(1.0, np.abs(z).max())
    gt = _torch_f64(lambda x: Fn.gelu(x, approximate="tanh"), z)
    assert np.abs(O.act("gelu_tanh", z) - gt).max() <= 1e-14 * max(1.0, np.abs(z).max())
    ge = _torch_f64(lambda x: Fn.gelu(x, approximate="none"), z)
    assert np.abs(O.act("gelu_erf", z) - ge).max() <= 1e-14 * max(1.0, np.abs(z).max())
    for name, fn, grad in (("silu", Fn.silu, O.silu_grad),
                           ("gelu_tanh", lambda x: Fn.gelu(x, approximate="tanh"),
                            lambda v: O.act_grad("gelu_tanh", v)),
                           ("gelu_erf", lambda x: Fn.gelu(x, approximate="none"),
                            lambda v: O.act_grad("gelu_erf", v))):
        x = torch.tensor(z, dtype=torch.float64, requires_grad=True)
        (g,) = torch.autograd.grad(fn(x).sum(), x)
        assert np.abs(grad(z) - g.numpy()).max() <= 1e-13, name
    # the planted mistake this catches: a GeLU-tanh with a cubic coefficient 1e-4 off
    c = 0.044715 + 1e-4
    wrong = 0.5 * z * (1 + np.tanh(math.sqrt(2 / math.pi) * (z + c * z ** 3)))
    assert np.abs(wrong - gt).max() > 1e-6


# ---------------------------------------------------------------------------
# Attention.
# ---------------------------------------------------------------------------

def test_attention_special_cases():
    rng = np.random.default_rng(3)
    V1 = rng.normal(size=(1, 4))
    o, p, _ = O.attention_head_forward(rng.normal(size=(1, 4)), rng.normal(size=(1, 4)), V1, True, 0.5)
    assert np.array_equal(p, np.ones((1, 1))) and np.allclose(o, V1, rtol=0, atol=0)
    N = 6
    Q, K, V = rng.normal(size=(N, 4)), rng.normal(size=(N, 4)), rng.normal(size=(N, 4))
    o, p, lse = O.attention_head_forward(Q, K, V, True, 0.5)
    assert np.allclose(o[0], V[0], rtol=0, atol=1e-15)
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-15) and np.all(np.triu(p, 1) == 0)
    # uniform scores: each row averages the visible value rows
    o, _, lse = O.attention_head_forward(np.zeros((N, 4)), K, V, True, 0.5)
    for r in range(N):
        assert np.allclose(o[r], V[:r + 1].mean(axis=0), atol=1e-14)
        assert abs(lse[r] - math.log(r + 1)) < 1e-14
    o, _, _ = O.attention_head_forward(np.zeros((N, 4)), K, V, False, 0.5)
    assert np.allclose(o, V.mean(axis=0)[None, :], atol=1e-14)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("t", [1, 2])
def test_attention_finite_differences(causal, t):
    rng = np.random.default_rng(21)
    N, nh, dh = 5, 2, 2
    d = nh * dh
    Xn = rng.normal(size=(N, d)); Wqkv = rng.normal(size=(d, 3 * d)); bqkv = rng.normal(size=3 * d)
    Wo = rng.normal(size=(d, d)); bo = rng.normal(size=d); G = rng.normal(size=(N, d))
    sc = 1 / math.sqrt(dh)
    U = O.attn_forward_unsplit(Xn, Wqkv, bqkv, Wo, bo, nh, dh, causal, sc)
    S = O.attn_forward_sharded(Xn, Wqkv, bqkv, Wo, bo, nh, dh, causal, sc, t)
    assert np.abs(U["Y"] - S["Y"]).max() < 1e-12
    loss = lambda: float((O.attn_forward_sharded(Xn, Wqkv, bqkv, Wo, bo, nh, dh, causal, sc, t)["Y"] * G).sum())
    b = O.attn_backward_sharded(G, Xn, Wqkv, Wo, S, nh, dh, sc, t)
    bu = O.attn_backward_unsplit(G, Xn, Wqkv, Wo, U, nh, dh, sc)
    for k in ("dXn", "dW_qkv", "db_qkv", "dW_o", "db_o"):
        assert np.abs(b[k] - bu[k]).max() < 1e-12
    _fd_check(loss, {"X": Xn, "W_qkv": Wqkv, "b_qkv": bqkv, "W_o": Wo, "b_o": bo},
              {"X": b["dXn"], "W_qkv": b["dW_qkv"], "b_qkv": b["db_qkv"], "W_o": b["dW_o"], "b_o": b["db_o"]})


# ---------------------------------------------------------------------------
# LayerNorm, SP LayerNorm, all-gather / reduce-scatter emulation.
# ---------------------------------------------------------------------------

def test_layernorm_special_cases():
    rng = np.random.default_rng(5)
    h = 6
    gamma, beta = rng.normal(size=h), rng.normal(size=h)
    x = np.full((2, h), 3.25)
    y, m, r = O.layernorm_forward(x, gamma, beta, 1e-5)
    assert np.allclose(y, np.broadcast_to(beta, y.shape), rtol=0, atol=0)
    x = rng.normal(size=(4, h)); dy = rng.normal(size=(4, h))
    y, m, r = O.layernorm_forward(x, gamma, beta, 1e-5)
    assert np.allclose(((y - beta) / gamma).mean(axis=1), 0, atol=1e-14)
    dx, dg, db = O.layernorm_backward(dy, x, gamma, m, r)
    assert np.allclose(dx.sum(axis=1), 0, atol=1e-12)   # a shift of x leaves y unchanged


def test_layernorm_finite_differences():
    rng = np.random.default_rng(6)
    s, h = 3, 6
    x, gamma, beta, G = rng.normal(size=(s, h)), rng.normal(size=h), rng.normal(size=h), rng.normal(size=(s, h))
    loss = lambda: float((O.layernorm_forward(x, gamma, beta, 1e-5)[0] * G).sum())
    y, m, r = O.layernorm_forward(x, gamma, beta, 1e-5)
    dx, dg, db = O.layernorm_backward(G, x, gamma, m, r)
    _fd_check(loss, {"x": x, "gamma": gamma, "beta": beta}, {"x": dx, "gamma": dg, "beta": db})


@pytest.mark.parametrize("t", [1, 2, 4])
def test_sp_layernorm_and_collectives(t):
    rng = np.random.default_rng(8)
    s, h = 8, 6
    X = rng.normal(size=(s, h)); gamma, beta = rng.normal(size=h), rng.normal(size=h)
    dY = rng.normal(size=(s, h))
    Xs = X.reshape(t, s // t, h)
    ys, ms, rs = O.sp_layernorm_forward(Xs, gamma, beta, 1e-5)
    y, m, r = O.layernorm_forward(X, gamma, beta, 1e-5)
    assert np.array_equal(O.all_gather_seq(ys), y)
    dxs, dgp, dbp, dg, db = O.sp_layernorm_backward(dY.reshape(t, s // t, h), Xs, gamma, ms, rs)
    dx, dg_full, db_full = O.layernorm_backward(dY, X, gamma, m, r)
    assert np.allclose(dxs.reshape(s, h), dx, atol=1e-13)
    assert np.allclose(dg, dg_full, atol=1e-13) and np.allclose(db, db_full, atol=1e-13)
    assert np.allclose(dgp.sum(axis=0), dg, atol=1e-13)
    # reduce-scatter followed by all-gather is an all-reduce (same volume)
    parts = [rng.normal(size=(s, h)) for _ in range(t)]
    assert np.allclose(O.all_gather_seq(O.reduce_scatter_seq(parts, t)), sum(parts), atol=1e-13)


# ---------------------------------------------------------------------------
# Whole layer: SP form equals the replicated form; gradients by FD.
# ---------------------------------------------------------------------------

def _tiny_layer(rng, s=4, d=4, F=8):
    p = {"ln1_g": 1 + 0.1 * rng.normal(size=d), "ln1_b": 0.1 * rng.normal(size=d),
         "W_qkv": rng.normal(size=(d, 3 * d)), "b_qkv": rng.normal(size=3 * d),
         "W_o": rng.normal(size=(d, d)), "b_o": rng.normal(size=d),
         "ln2_g": 1 + 0.1 * rng.normal(size=d), "ln2_b": 0.1 * rng.normal(size=d),
         "W_up": rng.normal(size=(d, F)), "b_up": rng.normal(size=F),
         "W_down": rng.normal(size=(F, d)), "b_down": rng.normal(size=d)}
    cfg = {"n_heads": 2, "head_dim": d // 2, "causal": True, "scale": 1 / math.sqrt(d // 2),
           "eps": 1e-5, "act": "gelu_tanh"}
    return p, cfg


@pytest.mark.parametrize("sp", [False, True])
def test_layer_finite_differences(sp):
    rng = np.random.default_rng(31)
    t, s, d = 2, 4, 4
    p, cfg = _tiny_layer(rng, s, d)
    X = rng.normal(size=(s, d)); G = rng.normal(size=(s, d))
    Xin = X.reshape(t, s // t, d) if sp else X
    Gin = G.reshape(t, s // t, d) if sp else G
    fwd = O.layer_forward(Xin, p, cfg, t, sp)
    if sp:
        ref = O.layer_forward(X, p, cfg, t, False)
        assert np.abs(fwd["Y"].reshape(s, d) - ref["Y"]).max() < 1e-12
    g = O.layer_backward(Gin, Xin, p, cfg, t, fwd, sp)
    loss = lambda: float((O.layer_forward(Xin, p, cfg, t, sp)["Y"] * Gin).sum())
    params = {"X": Xin}
    params.update(p)
    grads = {"X": g["dX"]}
    grads.update({k: g[k] for k in p})
    _fd_check(loss, params, grads)


# ---------------------------------------------------------------------------
# Packing: plain element loops define each shard; pack/unpack is a bijection.
# ---------------------------------------------------------------------------

def test_packing_by_element_loops():
    rng = np.random.default_rng(9)
    h, F, t = 6, 8, 2
    W = rng.integers(0, 65535, size=(h, F)).astype(np.uint16)
    Pc = O.pack_col_weight(W, t)
    for i in range(t):
        for f in range(F // t):
            for k in range(h):
                assert Pc[i, f, k] == W[k, i * (F // t) + f]
    assert np.array_equal(O.unpack_col_weight(Pc), W)
    Wd = rng.integers(0, 65535, size=(F, h)).astype(np.uint16)
    Pr = O.pack_row_weight(Wd, t)
    for i in range(t):
        for c in range(h):
            for f in range(F // t):
                assert Pr[i, c, f] == Wd[i * (F // t) + f, c]
    assert np.array_equal(O.unpack_row_weight(Pr), Wd)
    # SwiGLU: shard i, group q, part (0 gate / 1 up), row r = column i*Ft + q*g + r
    g = 2
    Wg = rng.integers(0, 65535, size=(h, F)).astype(np.uint16)
    Ps = O.pack_swiglu_weight(Wg, W, t, group=g)
    Ft = F // t
    for i in range(t):
        for q in range(Ft // g):
            for r in range(g):
                col = i * Ft + q * g + r
                assert np.array_equal(Ps[i, q, 0, r], Wg[:, col])
                assert np.array_equal(Ps[i, q, 1, r], W[:, col])
    # QKV by head: shard i, local row = part*(d/t) + jj*dh + e  <->  column part*d + (i*nh/t + jj)*dh + e
    nh, dh, d = 4, 2, 8
    Wq = rng.integers(0, 65535, size=(d, 3 * d)).astype(np.uint16)
    Pq = O.pack_qkv_weight(Wq, nh, dh, t)
    for i in range(t):
        for part in range(3):
            for jj in range(nh // t):
                for e in range(dh):
                    row = part * (d // t) + jj * dh + e
                    col = part * d + (i * nh // t + jj) * dh + e
                    assert np.array_equal(Pq[i, row], Wq[:, col])


def test_bf16_conversion():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x4049, 0x7F80, 0x0001], dtype=np.uint16)
    v = O.bf16_to_f64(bits)
    assert v[0] == 1.0 and v[1] == -1.0 and v[2] == 0.0 and v[3] == 3.140625 and np.isinf(v[4])
    assert v[5] == 2.0 ** -133
    # round-to-nearest-even: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1.0)
    assert O.f64_to_bf16_bits(np.array([1 + 2 ** -8]))[0] == 0x3F80
    assert O.f64_to_bf16_bits(np.array([1 + 3 * 2 ** -8]))[0] == 0x3F82


def test_layer_forward_rows_matches_full_layer():
    rng = np.random.default_rng(32)
    p, cfg = _tiny_layer(rng, s=6, d=4)
    X = rng.normal(size=(6, 4))
    full = O.layer_forward(X, p, cfg, 2, False)
    rows = [0, 3, 5]
    part = O.layer_forward_rows(X, p, cfg, 2, rows)
    assert np.array_equal(part["X1"], full["X1"][rows])
    assert np.abs(part["Y"] - full["Y"][rows]).max() < 1e-13
