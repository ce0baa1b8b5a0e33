"""GPU parity of a full pre-LN TP transformer layer (replicated LayerNorms and
the sequence-parallel form) against the fp64 oracle, through the C ABI:
X1 = X + Attn(LN1(X)), Y = X1 + MLP(LN2(X1)), and every gradient."""

import math

import numpy as np
import pytest
import torch

import oracle as O
from megatron_tensor_transformer_shard_gb300 import _lib as L
from megatron_tensor_transformer_shard_gb300 import inputs as I
from megatron_tensor_transformer_shard_gb300 import tp as T

from gpu_helpers import assert_close, f64

pytestmark = pytest.mark.gpu

PARAMS = ("ln1_g", "ln1_b", "W_qkv", "b_qkv", "W_o", "b_o", "ln2_g", "ln2_b", "W_up", "b_up", "W_down", "b_down")


def _cfg(nh):
    return {"n_heads": nh, "head_dim": 128, "causal": True, "scale": 1.0 / math.sqrt(128), "eps": 1e-5,
            "act": "gelu_tanh"}


def _run_gpu(inp, nh, t, sp):
    dev = {k: v.cuda() for k, v in inp.items()}
    w = T.LayerWeights(dev, nh, 128, t)
    Y, saved = T.layer_forward(dev["X"], w, sp=sp)
    g = T.layer_backward(dev["dY"], saved, w)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    return Y, saved, g


@pytest.mark.parametrize("N,d,F,t,sp", [(256, 512, 2048, 2, False), (320, 512, 1024, 4, True),
                                        (512, 1024, 4096, 8, True), (200, 256, 1024, 2, False)])
def test_layer_parity(N, d, F, t, sp):
    nh = d // 128
    inp = I.layer_inputs(N, d, F, seed=11)
    Y, saved, g = _run_gpu(inp, nh, t, sp)
    ref = {k: f64(v) for k, v in inp.items()}
    p = {k: ref[k] for k in PARAMS}
    cfg = _cfg(nh)
    X, G = ref["X"], ref["dY"]
    if sp:
        X, G = X.reshape(t, N // t, d), G.reshape(t, N // t, d)
    fwd = O.layer_forward(X, p, cfg, t, sp)
    bwd = O.layer_backward(G, X, p, cfg, t, fwd, sp)
    assert_close("Y", f64(Y), fwd["Y"].reshape(N, d))
    assert_close("X1", f64(saved["X1"]), fwd["X1"].reshape(N, d))
    assert_close("dX", f64(g["dX"]), bwd["dX"].reshape(N, d))
    assert_close("dW_qkv", f64(g["Wqkv_p"]), O.pack_qkv_weight(bwd["W_qkv"], nh, 128, t))
    assert_close("db_qkv", f64(g["bqkv_p"]), O.pack_qkv_bias(bwd["b_qkv"], nh, 128, t))
    assert_close("dW_o", f64(g["Wo_p"]), O.pack_row_weight(bwd["W_o"], t))
    assert_close("db_o", f64(g["b_o"]), bwd["b_o"])
    assert_close("dW_up", f64(g["Wup_p"]), O.pack_col_weight(bwd["W_up"], t))
    assert_close("db_up", f64(g["b_up"]), bwd["b_up"])
    assert_close("dW_down", f64(g["Wdown_p"]), O.pack_row_weight(bwd["W_down"], t))
    assert_close("db_down", f64(g["b_down"]), bwd["b_down"])
    for k in ("ln1_g", "ln1_b", "ln2_g", "ln2_b"):
        assert_close("d" + k, f64(g[k]), bwd[k])
    if sp:  # each sequence shard's own LayerNorm weight-grad partial, before the sum
        _, m, r = O.sp_layernorm_forward(fwd["X1"], p["ln2_g"], p["ln2_b"], 1e-5)
        mg = O.mlp_backward_sharded(G.reshape(N, d), fwd["Xn2"], p["W_up"], p["W_down"], fwd["mlp"], "gelu_tanh", t)
        dxn2 = O.reduce_scatter_seq(mg["dX_partials"], t)
        _, dgp, _, _, _ = O.sp_layernorm_backward(dxn2, fwd["X1"], p["ln2_g"], m, r)
        assert_close("dln2_g partials", f64(g["ln2_g_part"]), dgp)


def _full_size(name):
    """The full-size layer in the launch configuration the bench times, against the fp64
    oracle on every row: forward (Y, X1), the gradient entering the attention block (dX1),
    and every gradient through attention and both LayerNorms (dX, dW_qkv, db_qkv, dW_o,
    db_o, dgamma / dbeta of both LayerNorms).  The MLP's own weight gradients are checked
    on sampled hidden units (whole columns need every token, which the oracle has here)."""
    c = I.CONFIGS[name]
    N, d, F, t, nh, sp = c["N"], c["d"], c["F"], c["t"], c["n_heads"], c["sp"]
    inp = I.layer_inputs(N, d, F, seed=0)
    Y, saved, g = _run_gpu(inp, nh, t, sp)
    ref = {k: f64(v) for k, v in inp.items()}
    del inp
    p = {k: ref[k] for k in PARAMS}
    cfg = _cfg(nh)
    eps, sc = cfg["eps"], cfg["scale"]
    X, G = ref["X"], ref["dY"]
    errs = {}
    # Forward on every row.  The sequence-parallel form only regroups the rows of the
    # LayerNorms and residual adds ([t][s/t][h] is [s][h]), so the replicated form gives
    # the same values row by row.
    Xn1, m1, r1 = O.layernorm_forward(X, p["ln1_g"], p["ln1_b"], eps)
    at = O.attn_forward_sharded(Xn1, p["W_qkv"], p["b_qkv"], p["W_o"], p["b_o"], nh, 128, True, sc, t)
    X1 = X + at["Y"]
    Xn2, m2, r2 = O.layernorm_forward(X1, p["ln2_g"], p["ln2_b"], eps)
    ml = O.mlp_forward_sharded(Xn2, p["W_up"], p["b_up"], p["W_down"], p["b_down"], "gelu_tanh", t)
    errs["Y"] = assert_close("Y", f64(Y).reshape(N, d), X1 + ml["Y"])
    errs["X1"] = assert_close("X1", f64(saved["X1"]).reshape(N, d), X1)
    # Backward: the MLP branch's input gradient, then LN2, then the attention block.
    mb = O.mlp_backward_sharded(G, Xn2, p["W_up"], p["W_down"], ml, "gelu_tanh", t, weight_grads=False)
    dx2, dg2, db2 = O.layernorm_backward(mb["dX"], X1, p["ln2_g"], m2, r2)
    dX1 = G + dx2
    errs["dX1"] = assert_close("dX1", f64(g["dX1"]).reshape(N, d), dX1)
    errs["dln2_g"] = assert_close("dln2_g", f64(g["ln2_g"]), dg2)
    errs["dln2_b"] = assert_close("dln2_b", f64(g["ln2_b"]), db2)
    fs = [0, 129, F // t - 1, F // t + 5, F // 2 + 7, F - 1]      # sampled hidden units
    Ft = F // t
    dZc = np.stack([mb["dZ"][f // Ft][:, f % Ft] for f in fs], axis=1)
    Ac = np.stack([ml["A"][f // Ft][:, f % Ft] for f in fs], axis=1)
    gu = g["Wup_p"].reshape(F, d)                                 # packed [t][Ft][d] == dW_up^T
    errs["dW_up cols"] = assert_close("dW_up columns", f64(gu[fs]).T, Xn2.T @ dZc)
    gd = g["Wdown_p"].cpu()                                       # [t][d][Ft]
    errs["dW_down rows"] = assert_close("dW_down rows", np.stack([f64(gd[f // Ft, :, f % Ft]) for f in fs]),
                                        Ac.T @ G)
    errs["db_up sampled"] = assert_close("db_up sampled", f64(g["b_up"])[fs], dZc.sum(axis=0))
    del mb, ml
    ab = O.attn_backward_sharded(dX1, Xn1, p["W_qkv"], p["W_o"], at, nh, 128, sc, t)
    dx1, dg1, db1 = O.layernorm_backward(ab["dXn"], X, p["ln1_g"], m1, r1)
    errs["dX"] = assert_close("dX", f64(g["dX"]).reshape(N, d), dX1 + dx1)
    errs["dW_qkv"] = assert_close("dW_qkv", f64(g["Wqkv_p"]), O.pack_qkv_weight(ab["dW_qkv"], nh, 128, t))
    errs["db_qkv"] = assert_close("db_qkv", f64(g["bqkv_p"]), O.pack_qkv_bias(ab["db_qkv"], nh, 128, t))
    errs["dW_o"] = assert_close("dW_o", f64(g["Wo_p"]), O.pack_row_weight(ab["dW_o"], t))
    errs["db_o"] = assert_close("db_o", f64(g["b_o"]), ab["db_o"])
    errs["dln1_g"] = assert_close("dln1_g", f64(g["ln1_g"]), dg1)
    errs["dln1_b"] = assert_close("dln1_b", f64(g["ln1_b"]), db1)
    print(f"\n{name} max|gpu-oracle|/max|oracle|: " + ", ".join(f"{k} {v:.2e}" for k, v in errs.items()))


@pytest.mark.slow
def test_full_layer_replicated_ln():
    """96 heads x 128, d = 12288, 2048 tokens, MLP 4d, t = 8."""
    _full_size("c4")


@pytest.mark.slow
def test_full_layer_sequence_parallel():
    """64 heads x 128, h = 8192, s = 4096, MLP 4h, t = 8, SP LayerNorms."""
    _full_size("c5")
