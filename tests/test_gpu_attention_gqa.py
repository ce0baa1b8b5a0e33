"""GPU parity of head-sharded attention with grouped-query heads (sharded by KV
group, KV heads replicated when n_kv < t), forward and backward, against the
fp64 oracle through the C ABI (max|gpu - oracle| <= 1e-2 max|oracle| per tensor),
and of the replica-group reduction of the W_qkv gradient."""

import math

import numpy as np
import pytest
import torch

import oracle as O
from megatron_tensor_transformer_shard_gb300 import _lib as L
from megatron_tensor_transformer_shard_gb300 import inputs as I

from gpu_helpers import assert_close, f64

pytestmark = pytest.mark.gpu

HD = 128


def _run(N, nh, nkv, t, causal, seed=0, bias=True):
    d = nh * HD
    inp = I.gqa_attn_inputs(N, d, nh, nkv, HD, bias=bias, seed=seed)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    kv_t = nkv // t if nkv >= t else 1
    R = (nh // t + 2 * kv_t) * HD
    bf16, f32 = torch.bfloat16, torch.float32
    Wqkv = torch.empty(t, R, d, dtype=bf16, device="cuda")
    L.tp_pack_qkv_gqa(dev["W_qkv"], d, nh, nkv, HD, t, Wqkv)
    bqkv = None
    if bias:
        bqkv = torch.empty(t, R, dtype=bf16, device="cuda")
        L.tp_pack_qkv_gqa_bias(dev["b_qkv"], nh, nkv, HD, t, bqkv)
    Wo = torch.empty(t, d, d // t, dtype=bf16, device="cuda")
    L.tp_pack_row(dev["W_o"], d, d, t, Wo)
    sc = 1.0 / math.sqrt(HD)
    Y = torch.empty(N, d, dtype=bf16, device="cuda")
    QKV = torch.empty(t, N, R, dtype=torch.float16, device="cuda")
    Od = torch.empty(t, N, d // t, dtype=bf16, device="cuda")
    lse = torch.empty(t, nh // t, N, dtype=f32, device="cuda")
    L.tp_attn_gqa_forward(dev["X"], N, d, nh, nkv, HD, t, int(causal), sc, Wqkv, bqkv, Wo, dev["b_o"], None, Y, QKV,
                          Od, lse, 0, None, 0)
    dX = torch.empty(N, d, dtype=bf16, device="cuda")
    dWq = torch.empty(t, R, d, dtype=f32, device="cuda")
    dbq = torch.empty(t, R, dtype=f32, device="cuda") if bias else None
    dWo = torch.empty(t, d, d // t, dtype=f32, device="cuda")
    dbo = torch.empty(d, dtype=f32, device="cuda") if bias else None
    nws = L.tp_attn_gqa_backward_workspace_size(N, d, nh, nkv, HD, t, 0)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    L.tp_attn_gqa_backward(dev["dY"], dev["X"], QKV, Od, lse, N, d, nh, nkv, HD, t, int(causal), sc, Wqkv, Wo, dX,
                           dWq, dbq, dWo, dbo, 0, 0, ws, nws)
    dW_full = torch.empty(d, (nh + 2 * nkv) * HD, dtype=f32, device="cuda")
    L.tp_reduce_qkv_gqa_grad(dWq, d, nh, nkv, HD, t, dW_full, 0)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    ref = {k: (f64(v) if v is not None else None) for k, v in inp.items()}
    fw = O.attn_gqa_forward_sharded(ref["X"], ref["W_qkv"], ref["b_qkv"], ref["W_o"], ref["b_o"], nh, nkv, HD,
                                    causal, sc, t)
    bw = O.attn_gqa_backward_sharded(ref["dY"], ref["X"], ref["W_qkv"], ref["W_o"], fw, nh, nkv, HD, sc, t)
    return dict(Y=Y, QKV=QKV, O=Od, dX=dX, dWq=dWq, dbq=dbq, dWo=dWo, dbo=dbo, dW_full=dW_full), fw, bw, R


@pytest.mark.parametrize("nh,nkv,t,causal", [
    (8, 2, 2, True),    # GQA, two KV heads, one per shard
    (8, 2, 4, True),    # each KV head replicated on two shards
    (8, 1, 4, False),   # MQA, replicated four times, non-causal
    (8, 4, 2, False),   # two KV heads per shard
    (8, 8, 2, True),    # multi-head through the grouped-query path
])
def test_attention_gqa_parity(nh, nkv, t, causal):
    N = 300  # three query/key blocks of 128, ragged tail
    g, fw, bw, R = _run(N, nh, nkv, t, causal, seed=nh + nkv + t)
    assert_close("Y", f64(g["Y"]), fw["Y"])
    qkv = g["QKV"].cpu().double().numpy()
    for i in range(t):
        assert_close(f"QKV[{i}]", qkv[i], fw["QKV"][i])
        assert_close(f"O[{i}]", f64(g["O"][i]), fw["O"][i])
    assert_close("dX", f64(g["dX"]), bw["dXn"])
    for i in range(t):
        assert_close(f"dWqkv copy {i}", f64(g["dWq"][i]), bw["dWqkv_shard"][i].T)
        assert_close(f"dbqkv copy {i}", f64(g["dbq"][i]), bw["dbqkv_shard"][i])
    assert_close("dW_qkv (copies summed)", f64(g["dW_full"]), bw["dW_qkv"])
    d = nh * HD
    dWo_unpacked = np.concatenate([f64(g["dWo"][i]).T for i in range(t)], axis=0)
    assert_close("dW_o", dWo_unpacked, bw["dW_o"])
    assert_close("db_o", f64(g["dbo"]), bw["db_o"])


def test_mha_entry_points_agree_with_gqa_path():
    """tp_attn_forward is the grouped-query call with n_kv = n_heads: same bits."""
    N, nh, t = 200, 8, 2
    d = nh * HD
    inp = I.attn_inputs(N, d, bias=True, dy=False, seed=3, device="cuda")
    R = 3 * d // t
    Wqkv = torch.empty(t, R, d, dtype=torch.bfloat16, device="cuda")
    L.tp_pack_qkv_heads(inp["W_qkv"], d, nh, HD, t, Wqkv)
    Wqkv2 = torch.empty_like(Wqkv)
    L.tp_pack_qkv_gqa(inp["W_qkv"], d, nh, nh, HD, t, Wqkv2)
    torch.cuda.synchronize()
    assert torch.equal(Wqkv.view(torch.int16), Wqkv2.view(torch.int16))
    Wo = torch.empty(t, d, d // t, dtype=torch.bfloat16, device="cuda")
    L.tp_pack_row(inp["W_o"], d, d, t, Wo)
    outs = []
    for gqa in (False, True):
        Y = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
        QKV = torch.empty(t, N, R, dtype=torch.float16, device="cuda")
        Od = torch.empty(t, N, d // t, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(t, nh // t, N, dtype=torch.float32, device="cuda")
        if gqa:
            L.tp_attn_gqa_forward(inp["X"], N, d, nh, nh, HD, t, 1, 0.1, Wqkv, None, Wo, None, None, Y, QKV, Od, lse,
                                  0, None, 0)
        else:
            L.tp_attn_forward(inp["X"], N, d, nh, HD, t, 1, 0.1, Wqkv, None, Wo, None, None, Y, QKV, Od, lse, 0, None, 0)
        outs.append(Y)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_reduce_gqa_grad_is_unpack_without_replicas():
    nh, nkv, t, d = 8, 8, 4, 256
    R = (nh // t + 2 * (nkv // t)) * HD
    g = torch.Generator().manual_seed(5)
    dWp = torch.randn(t, R, d, generator=g).cuda()
    out = torch.empty(d, (nh + 2 * nkv) * HD, device="cuda")
    L.tp_reduce_qkv_gqa_grad(dWp, d, nh, nkv, HD, t, out, 0)
    torch.cuda.synchronize()
    # each column appears in exactly one shard: out^T gathers rows of dWp
    for i in range(t):
        cols = O.gqa_qkv_shard_columns(nh, nkv, HD, t, i)
        assert torch.equal(out[:, torch.as_tensor(cols).cuda()].T.contiguous(), dWp[i])
