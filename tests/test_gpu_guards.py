"""Out-of-bounds write detection, the stand-in for a memory checker (which this GPU pool
does not run): every output and workspace of the library's entry points sits between
4 KB guard regions filled with a known byte, at ragged shapes whose last tiles, rows or
columns are partial; after the call the guards must be unchanged.  (The MLP GEMMs, both
split-K forms and the allocation-free column sum have guarded tests of their own.)"""

import math

import numpy as np
import pytest
import torch

from megatron_tensor_transformer_shard_gb300 import _lib as L
from megatron_tensor_transformer_shard_gb300 import inputs as I
from megatron_tensor_transformer_shard_gb300 import tp as T

from gpu_helpers import Guarded, guarded_ws

pytestmark = pytest.mark.gpu

BF, H, F32 = torch.bfloat16, torch.float16, torch.float32


def _done(*guards):
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    for name, g in guards:
        g.check(name)


def _packed_attn(N, nh, t, seed, f16):
    dh = 128
    d = nh * dh
    inp = I.attn_inputs(N, d, bias=True, dy=True, seed=seed)
    dev = {k: v.cuda() for k, v in inp.items()}
    Wq = torch.empty(t, 3 * d // t, d, dtype=BF, device="cuda")
    bq = torch.empty(t, 3 * d // t, dtype=BF, device="cuda")
    Wo = torch.empty(t, d, d // t, dtype=BF, device="cuda")
    L.tp_pack_qkv_heads(dev["W_qkv"], d, nh, dh, t, Wq)
    L.tp_pack_qkv_bias(dev["b_qkv"], d, nh, dh, t, bq)
    L.tp_pack_row(dev["W_o"], d, d, t, Wo)
    X = dev["X"]
    if f16:
        W16 = torch.empty(Wq.shape, dtype=H, device="cuda")
        L.tp_convert_bf16_to_f16(Wq, Wq.numel(), W16)
        Wq, X = W16, X.to(H)
    return dev, X, Wq, bq, Wo, d


@pytest.mark.parametrize("f16", [False, True])
@pytest.mark.parametrize("N,nh,t", [(333, 4, 2), (200, 8, 8)])
def test_attention_block_writes_stay_inside(N, nh, t, f16):
    dev, X, Wq, bq, Wo, d = _packed_attn(N, nh, t, 100 + N, f16)
    flag = L.TP_ATTN_F16_INPUT if f16 else 0
    sc = 1 / math.sqrt(128)
    Y, QKV = Guarded((N, d), BF), Guarded((t, N, 3 * d // t), H)
    O, lse = Guarded((t, N, d // t), BF), Guarded((t, nh // t, N), F32)
    naw = L.tp_attn_forward_workspace_size(N, d, nh, 128, t, flag)
    aws = guarded_ws(naw)
    L.tp_attn_forward(X, N, d, nh, 128, t, 1, sc, Wq, bq, Wo, dev["b_o"], dev["X"], Y.t, QKV.t, O.t, lse.t, flag,
                      aws.t, naw)
    _done(("Y", Y), ("QKV", QKV), ("O", O), ("lse", lse), ("forward ws", aws))
    dX = Guarded((N, d), BF)
    dWq, dbq = Guarded((t, 3 * d // t, d), F32), Guarded((t, 3 * d // t), F32)
    dWo, dbo = Guarded((t, d, d // t), F32), Guarded((d,), F32)
    nws = L.tp_attn_backward_workspace_size(N, d, nh, 128, t, flag)
    ws = guarded_ws(nws)
    L.tp_attn_backward(dev["dY"], X, QKV.t, O.t, lse.t, N, d, nh, 128, t, 1, sc, Wq, Wo, dX.t, dWq.t, dbq.t, dWo.t,
                       dbo.t, 0, flag, ws.t, nws)
    _done(("dX", dX), ("dW_qkv", dWq), ("db_qkv", dbq), ("dW_o", dWo), ("db_o", dbo), ("backward ws", ws))
    assert torch.isfinite(dX.t.float()).all() and torch.isfinite(dWq.t).all()


def test_attention_core_writes_stay_inside():
    N, nh, t = 333, 4, 2
    dev, X, Wq, bq, Wo, d = _packed_attn(N, nh, t, 7, False)
    sc = 1 / math.sqrt(128)
    QKV = torch.empty(t, N, 3 * d // t, dtype=H, device="cuda")
    Ot = torch.empty(t, N, d // t, dtype=BF, device="cuda")
    lt = torch.empty(t, nh // t, N, dtype=F32, device="cuda")
    L.tp_attn_forward(X, N, d, nh, 128, t, 1, sc, Wq, bq, Wo, None, None, torch.empty(N, d, dtype=BF, device="cuda"),
                      QKV, Ot, lt, 0, None, 0)
    O, lse = Guarded((t, N, d // t), BF), Guarded((t, nh // t, N), F32)
    L.tp_attn_core_forward(QKV, N, d, nh, nh, 128, t, 1, sc, O.t, lse.t)
    dO = (torch.randn(t, N, d // t, generator=torch.Generator().manual_seed(3)) * 0.1).to(H).cuda()
    Dv, dQKV = Guarded((t, nh // t, N), F32), Guarded((t, N, 3 * d // t), BF)
    L.tp_attn_core_backward(QKV, O.t, dO, lse.t, N, d, nh, nh, 128, t, 1, sc, Dv.t, dQKV.t)
    _done(("O", O), ("lse", lse), ("D", Dv), ("dQKV", dQKV))


def test_gqa_attention_writes_stay_inside():
    N, nh, nkv, t, dh = 333, 8, 2, 4, 128
    d = nh * dh
    inp = I.gqa_attn_inputs(N, d, nh, nkv, dh, bias=True, dy=True, seed=5)
    dev = {k: v.cuda() for k, v in inp.items()}
    kv_t = nkv // t if nkv >= t else 1
    R = (nh // t + 2 * kv_t) * dh
    Wq = torch.empty(t, R, d, dtype=BF, device="cuda")
    bq = torch.empty(t, R, dtype=BF, device="cuda")
    Wo = torch.empty(t, d, d // t, dtype=BF, device="cuda")
    L.tp_pack_qkv_gqa(dev["W_qkv"], d, nh, nkv, dh, t, Wq)
    L.tp_pack_qkv_gqa_bias(dev["b_qkv"], nh, nkv, dh, t, bq)
    L.tp_pack_row(dev["W_o"], d, d, t, Wo)
    sc = 1 / math.sqrt(dh)
    Y, QKV = Guarded((N, d), BF), Guarded((t, N, R), H)
    O, lse = Guarded((t, N, d // t), BF), Guarded((t, nh // t, N), F32)
    L.tp_attn_gqa_forward(dev["X"], N, d, nh, nkv, dh, t, 1, sc, Wq, bq, Wo, dev["b_o"], None, Y.t, QKV.t, O.t, lse.t,
                          0, None, 0)
    _done(("Y", Y), ("QKV", QKV), ("O", O), ("lse", lse))
    dX, dWq, dbq = Guarded((N, d), BF), Guarded((t, R, d), F32), Guarded((t, R), F32)
    dWo, dbo = Guarded((t, d, d // t), F32), Guarded((d,), F32)
    nws = L.tp_attn_gqa_backward_workspace_size(N, d, nh, nkv, dh, t, 0)
    ws = guarded_ws(nws)
    L.tp_attn_gqa_backward(dev["dY"], dev["X"], QKV.t, O.t, lse.t, N, d, nh, nkv, dh, t, 1, sc, Wq, Wo, dX.t, dWq.t,
                           dbq.t, dWo.t, dbo.t, 0, 0, ws.t, nws)
    _done(("dX", dX), ("dW_qkv", dWq), ("db_qkv", dbq), ("dW_o", dWo), ("db_o", dbo), ("ws", ws))


@pytest.mark.parametrize("s,h,t,f16", [(8 * 21, 4992, 8, False), (48, 1000 - 1000 % 8, 2, True), (3, 264, 1, False)])
def test_layernorm_writes_stay_inside(s, h, t, f16):
    inp = I.ln_inputs(s, h, seed=s)
    dev = {k: v.cuda() for k, v in inp.items()}
    Y, mean, rstd = Guarded((s, h), H if f16 else BF), Guarded((s,), F32), Guarded((s,), F32)
    fwd = L.tp_sp_layernorm_forward_f16 if f16 else L.tp_sp_layernorm_forward
    fwd(dev["X"], s, h, t, dev["gamma"], dev["beta"], 1e-5, Y.t, mean.t, rstd.t)
    _done(("Y", Y), ("mean", mean), ("rstd", rstd))
    dX = Guarded((s, h), BF)
    gp, bp, g, b = Guarded((t, h), F32), Guarded((t, h), F32), Guarded((h,), F32), Guarded((h,), F32)
    L.tp_sp_layernorm_backward(dev["dY"], dev["X"], dev["gamma"], mean.t, rstd.t, dev["X"], s, h, t, dX.t, gp.t, bp.t,
                               g.t, b.t)
    _done(("dX", dX), ("dgamma part", gp), ("dbeta part", bp), ("dgamma", g), ("dbeta", b))


@pytest.mark.parametrize("M,h,F,t", [(3, 264, 1024, 4), (1, 512, 2048, 2)])
def test_decode_swiglu_writes_stay_inside(M, h, F, t):
    inp = I.swiglu_inputs(M, h, F, seed=9)
    dev = {k: v.cuda() for k, v in inp.items()}
    Wgu = torch.empty(2 * F, h, dtype=BF, device="cuda")
    Wd = torch.empty(t, h, F // t, dtype=BF, device="cuda")
    L.tp_pack_swiglu(dev["W_gate"], dev["W_up"], h, F, t, Wgu)
    L.tp_pack_row(dev["W_down"], F, h, t, Wd)
    y, a = Guarded((M, h), BF), Guarded((M, F), BF)
    L.tp_decode_swiglu_forward(dev["X"], M, h, F, t, Wgu, Wd, y.t, a.t)
    _done(("y", y), ("a", a))


def test_decode_attention_writes_stay_inside():
    """One decode step: the new key / value go to position pos[b] of every cache copy and
    nowhere else; y and the workspace stay inside too."""
    B, nh, nkv, t, L_max, hd = 3, 8, 2, 4, 300, 128
    d = nh * hd
    inp = I.decode_attn_inputs(B, d, nh, nkv, hd, L_max, bias=True, seed=12)
    w = T.DecodeAttnWeights(inp["W_qkv"].cuda(), inp["b_qkv"].cuda(), inp["W_o"].cuda(), inp["b_o"].cuda(), nh, nkv,
                            hd, t)
    shape = w.cache_shape(B, L_max)
    K, V = Guarded(shape, H), Guarded(shape, H)
    K.t.normal_()
    V.t.normal_()
    pos = torch.tensor([0, 137, L_max - 1], dtype=torch.int32).cuda()
    nws = L.tp_decode_attn_workspace_size(B, d, nh, nkv, hd, t, L_max)
    ws = guarded_ws(nws)
    y = Guarded((B, d), BF)
    T.decode_attn_forward(inp["x"].cuda(), w, K.t, V.t, pos, ws=ws.t, out=y.t)
    _done(("K cache", K), ("V cache", V), ("ws", ws), ("y", y))


def test_embedding_writes_stay_inside():
    N, V, h, t = 1000, 96, 264, 4
    ids = I.token_ids(N, V, seed=1).cuda()
    inp = I.embedding_inputs(N, V, h, seed=2)
    Y = Guarded((N, h), BF)
    L.tp_vocab_embedding_forward(ids, N, V, h, t, inp["E"].cuda(), Y.t)
    dE = Guarded((V, h), F32, fill=torch.zeros(V, h))
    nws = L.tp_vocab_embedding_backward_workspace_size(N)
    ws = guarded_ws(nws)
    L.tp_vocab_embedding_backward(ids, inp["dY"].cuda(), N, V, h, t, dE.t, 1, ws.t, nws)
    _done(("Y", Y), ("dE", dE), ("ws", ws))


@pytest.mark.parametrize("rows,cols", [(333, 1026), (1, 8), (4100, 264)])
def test_colsum_and_shard_reduce_write_stay_inside(rows, cols):
    G = torch.randn(rows, cols, generator=torch.Generator().manual_seed(rows)).to(BF).cuda()
    out = Guarded((cols,), F32)
    nws = L.tp_colsum_workspace_size(rows, cols)
    ws = guarded_ws(nws)
    L.tp_colsum(G, rows, cols, out.t, 0, ws.t, nws)
    _done(("colsum out", out), ("colsum ws", ws))
    t = 3
    P = torch.randn(t, rows, cols - cols % 8, generator=torch.Generator().manual_seed(1)).cuda()
    c8 = cols - cols % 8
    yb, yf = Guarded((rows, c8), BF), Guarded((rows, c8), F32)
    L.tp_shard_reduce(P, rows, c8, t, None, None, yb.t, yf.t)
    _done(("shard sum bf16", yb), ("shard sum f32", yf))


def test_packing_writes_stay_inside():
    h, F, t = 40, 48, 2
    W = torch.randn(h, F).to(BF).cuda()
    Wp, back = Guarded((t, F // t, h), BF), Guarded((h, F), BF)
    L.tp_pack_col(W, h, F, t, Wp.t)
    L.tp_unpack_col(Wp.t, h, F, t, back.t)
    Wd = torch.randn(F, h).to(BF).cuda()
    Wdp = Guarded((t, h, F // t), BF)
    L.tp_pack_row(Wd, F, h, t, Wdp.t)
    nh, dh = 6, 64
    dq = nh * dh
    Wq = torch.randn(dq, 3 * dq).to(BF).cuda()
    Wqp = Guarded((3, 3 * dq // 3, dq), BF)
    L.tp_pack_qkv_heads(Wq, dq, nh, dh, 3, Wqp.t)
    conv = Guarded((1037,), H)
    L.tp_convert_bf16_to_f16(torch.randn(1037).to(BF).cuda(), 1037, conv.t)
    _done(("pack col", Wp), ("unpack col", back), ("pack row", Wdp), ("pack qkv", Wqp), ("bf16 -> fp16", conv))
    assert torch.equal(back.t, W)
