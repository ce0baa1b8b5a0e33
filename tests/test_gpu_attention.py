"""GPU parity of head-sharded causal attention (QKV column-parallel GEMM,
per-head flash attention on tcgen05, W_o row-parallel GEMM + g) against the
fp64 oracle, through the C ABI."""

import math

import numpy as np
import pytest
import torch

import oracle as O
from megatron_tensor_transformer_shard_gb300 import _lib as L
from megatron_tensor_transformer_shard_gb300 import inputs as I

from gpu_helpers import assert_close, f64

pytestmark = pytest.mark.gpu


def pack_attn(dev, d, nh, dh, t):
    Wqkv_p = torch.empty(t, 3 * d // t, d, dtype=torch.bfloat16, device="cuda")
    bqkv_p = torch.empty(t, 3 * d // t, dtype=torch.bfloat16, device="cuda")
    Wo_p = torch.empty(t, d, d // t, dtype=torch.bfloat16, device="cuda")
    L.tp_pack_qkv_heads(dev["W_qkv"], d, nh, dh, t, Wqkv_p)
    L.tp_pack_qkv_bias(dev["b_qkv"], d, nh, dh, t, bqkv_p)
    L.tp_pack_row(dev["W_o"], d, d, t, Wo_p)
    return Wqkv_p, bqkv_p, Wo_p


def run_fwd(N, nh, t, causal, seed=0, dh=128, scale=None):
    d = nh * dh
    inp = I.attn_inputs(N, d, bias=True, dy=True, seed=seed)
    dev = {k: v.cuda() for k, v in inp.items()}
    Wqkv_p, bqkv_p, Wo_p = pack_attn(dev, d, nh, dh, t)
    Y = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
    QKV = torch.empty(t, N, 3 * d // t, dtype=torch.float16, device="cuda")
    Osv = torch.empty(t, N, d // t, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(t, nh // t, N, dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(dh) if scale is None else scale
    L.tp_attn_forward(dev["X"], N, d, nh, dh, t, int(causal), scale, Wqkv_p, bqkv_p, Wo_p, dev["b_o"], None, Y, QKV,
                      Osv, lse, 0, None, 0)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    ref = {k: f64(v) for k, v in inp.items()}
    o = O.attn_forward_sharded(ref["X"], ref["W_qkv"], ref["b_qkv"], ref["W_o"], ref["b_o"], nh, dh, causal, scale, t)
    return dict(inp=inp, dev=dev, ref=ref, o=o, Y=Y, QKV=QKV, O=Osv, lse=lse, packed=(Wqkv_p, bqkv_p, Wo_p),
                d=d, scale=scale)


@pytest.mark.parametrize("N,nh,t,causal", [(256, 2, 2, True), (200, 4, 4, True), (128, 2, 1, False),
                                           (333, 4, 2, False), (1, 2, 2, True), (640, 8, 8, True)])
def test_attention_forward_parity(N, nh, t, causal):
    r = run_fwd(N, nh, t, causal)
    o = r["o"]
    assert_close("QKV", f64(r["QKV"]), np.stack(o["QKV"]))
    assert_close("O", f64(r["O"]), np.stack(o["O"]))
    assert_close("lse", f64(r["lse"]).reshape(nh, N), o["lse"])
    assert_close("Y", f64(r["Y"]), o["Y"])


@pytest.mark.parametrize("N,causal,scale", [(384, True, 4.0), (333, False, 4.0), (384, True, -0.5),
                                            (200, False, -0.5), (256, True, 0.0)])
def test_attention_forward_scales(N, causal, scale):
    """Logit spreads far beyond the default scale (the row maximum jumps many
    times, so O is rescaled often), a negative scale (the largest softmax weight
    sits at the smallest Q K^T entry) and scale 0 (uniform weights over the
    visible keys)."""
    nh, t = 4, 2
    r = run_fwd(N, nh, t, causal, seed=5, scale=scale)
    o = r["o"]
    assert_close("O", f64(r["O"]), np.stack(o["O"]))
    assert_close("lse", f64(r["lse"]).reshape(nh, N), o["lse"])
    assert_close("Y", f64(r["Y"]), o["Y"])


def _ws_dqkv(ws, N, d, nh, t):
    """dQKV inside the backward workspace (layout documented in include/tp.h)."""
    r = lambda v: (v + 255) // 256 * 256
    off = r(N * d * 2) + r(N * nh * 4)
    return ws[off:off + N * 3 * d * 2].view(torch.bfloat16).view(t, N, 3 * d // t)


@pytest.mark.parametrize("N,nh,t,causal", [(256, 2, 2, True), (200, 4, 4, True), (333, 4, 2, False),
                                           (128, 2, 1, True), (1, 2, 2, True), (640, 8, 8, True)])
def test_attention_backward_parity(N, nh, t, causal):
    dh = 128
    r = run_fwd(N, nh, t, causal, seed=3)
    d, dev, ref, o = r["d"], r["dev"], r["ref"], r["o"]
    Wqkv_p, _, Wo_p = r["packed"]
    dX = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
    dWqkv = torch.empty(t, 3 * d // t, d, dtype=torch.float32, device="cuda")
    dbqkv = torch.empty(t, 3 * d // t, dtype=torch.float32, device="cuda")
    dWo = torch.empty(t, d, d // t, dtype=torch.float32, device="cuda")
    dbo = torch.empty(d, dtype=torch.float32, device="cuda")
    nws = L.tp_attn_backward_workspace_size(N, d, nh, dh, t, 0)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    L.tp_attn_backward(dev["dY"], dev["X"], r["QKV"], r["O"], r["lse"], N, d, nh, dh, t, int(causal), r["scale"],
                       Wqkv_p, Wo_p, dX, dWqkv, dbqkv, dWo, dbo, 0, 0, ws, nws)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    b = O.attn_backward_sharded(ref["dY"], ref["X"], ref["W_qkv"], ref["W_o"], o, nh, dh, r["scale"], t)
    assert_close("dQKV", f64(_ws_dqkv(ws, N, d, nh, t)), np.stack(b["dQKV"]))
    assert_close("dX", f64(dX), b["dXn"])
    assert_close("dW_qkv (packed)", f64(dWqkv), O.pack_qkv_weight(b["dW_qkv"], nh, dh, t))
    assert_close("db_qkv (packed)", f64(dbqkv), O.pack_qkv_bias(b["db_qkv"], nh, dh, t))
    assert_close("dW_o (packed)", f64(dWo), O.pack_row_weight(b["dW_o"], t))
    assert_close("db_o", f64(dbo), b["db_o"])


@pytest.mark.parametrize("N,causal", [(333, True), (256, False)])
def test_attention_core_entry_points(N, causal):
    """tp_attn_core_forward / tp_attn_core_backward run the same kernels as the
    full attention block, so on the block's own saved QKV and dO they must give
    its O, lse and dQKV bit for bit (those are checked against the oracle above)."""
    nh, t, dh = 4, 2, 128
    r = run_fwd(N, nh, t, causal, seed=7)
    d, dev = r["d"], r["dev"]
    O2 = torch.empty_like(r["O"])
    lse2 = torch.empty_like(r["lse"])
    L.tp_attn_core_forward(r["QKV"], N, d, nh, nh, dh, t, int(causal), r["scale"], O2, lse2)
    torch.cuda.synchronize()
    assert torch.equal(O2, r["O"]) and torch.equal(lse2, r["lse"])

    Wqkv_p, _, Wo_p = r["packed"]
    nws = L.tp_attn_backward_workspace_size(N, d, nh, dh, t, 0)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    L.tp_attn_backward(dev["dY"], dev["X"], r["QKV"], r["O"], r["lse"], N, d, nh, dh, t, int(causal), r["scale"],
                       Wqkv_p, Wo_p, torch.empty(N, d, dtype=torch.bfloat16, device="cuda"),
                       torch.empty(t, 3 * d // t, d, dtype=torch.float32, device="cuda"), None,
                       torch.empty(t, d, d // t, dtype=torch.float32, device="cuda"), None, 0, 0, ws, nws)
    dO = ws[:N * d * 2].view(torch.float16).view(t, N, d // t)
    Dvec = torch.empty(t, nh // t, N, dtype=torch.float32, device="cuda")
    dQKV2 = torch.full((t, N, 3 * d // t), float("nan"), dtype=torch.bfloat16, device="cuda")
    L.tp_attn_core_backward(r["QKV"], r["O"], dO, r["lse"], N, d, nh, nh, dh, t, int(causal), r["scale"], Dvec, dQKV2)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    assert torch.equal(dQKV2, _ws_dqkv(ws, N, d, nh, t))


# ---------------------------------------------------------------------------
# The fp16 attention input (TP_ATTN_F16_INPUT): X and the packed W_qkv in IEEE fp16,
# dQKV in fp16 in the backward.  The oracle's inputs are the same values (bf16 -> fp16
# is exact for them), so the criterion is unchanged.
# ---------------------------------------------------------------------------

def test_convert_bf16_to_f16_exact():
    """bf16 values in fp16's normal range convert exactly; the ragged tail too."""
    g = torch.Generator().manual_seed(90)
    x = (torch.randn(1037, generator=g) * 3).to(torch.bfloat16)
    out = torch.empty(1037, dtype=torch.float16, device="cuda")
    L.tp_convert_bf16_to_f16(x.cuda(), x.numel(), out)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu().float(), x.float())


@pytest.mark.parametrize("N,nh,t,causal", [(256, 2, 2, True), (333, 4, 2, False), (640, 8, 8, True)])
def test_attention_f16_input_forward_backward(N, nh, t, causal):
    dh = 128
    d = nh * dh
    inp = I.attn_inputs(N, d, bias=True, dy=True, seed=91)
    dev = {k: v.cuda() for k, v in inp.items()}
    Wqkv_p, bqkv_p, Wo_p = pack_attn(dev, d, nh, dh, t)
    W16 = torch.empty(Wqkv_p.shape, dtype=torch.float16, device="cuda")
    L.tp_convert_bf16_to_f16(Wqkv_p, Wqkv_p.numel(), W16)
    X16 = dev["X"].to(torch.float16)
    flag = L.TP_ATTN_F16_INPUT
    scale = 1.0 / math.sqrt(dh)
    Y = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
    QKV = torch.empty(t, N, 3 * d // t, dtype=torch.float16, device="cuda")
    Osv = torch.empty(t, N, d // t, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(t, nh // t, N, dtype=torch.float32, device="cuda")
    naw = L.tp_attn_forward_workspace_size(N, d, nh, dh, t, flag)
    aws = torch.empty(naw, dtype=torch.uint8, device="cuda")
    L.tp_attn_forward(X16, N, d, nh, dh, t, int(causal), scale, W16, bqkv_p, Wo_p, dev["b_o"], None, Y, QKV, Osv, lse,
                      flag, aws, naw)
    dX = torch.empty(N, d, dtype=torch.bfloat16, device="cuda")
    dWqkv = torch.empty(t, 3 * d // t, d, dtype=torch.float32, device="cuda")
    dbqkv = torch.empty(t, 3 * d // t, dtype=torch.float32, device="cuda")
    dWo = torch.empty(t, d, d // t, dtype=torch.float32, device="cuda")
    dbo = torch.empty(d, dtype=torch.float32, device="cuda")
    nws = L.tp_attn_backward_workspace_size(N, d, nh, dh, t, flag)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    L.tp_attn_backward(dev["dY"], X16, QKV, Osv, lse, N, d, nh, dh, t, int(causal), scale, W16, Wo_p, dX, dWqkv, dbqkv,
                       dWo, dbo, 0, flag, ws, nws)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    ref = {k: f64(v) for k, v in inp.items()}
    o = O.attn_forward_sharded(ref["X"], ref["W_qkv"], ref["b_qkv"], ref["W_o"], ref["b_o"], nh, dh, causal, scale, t)
    assert_close("QKV", f64(QKV), np.stack(o["QKV"]))
    assert_close("O", f64(Osv), np.stack(o["O"]))
    assert_close("Y", f64(Y), o["Y"])
    b = O.attn_backward_sharded(ref["dY"], ref["X"], ref["W_qkv"], ref["W_o"], o, nh, dh, scale, t)
    off = ((N * d * 2 + 255) // 256) * 256 + ((N * nh * 4 + 255) // 256) * 256
    dqkv = ws[off:off + N * 3 * d * 2].view(torch.float16).view(t, N, 3 * d // t)
    assert_close("dQKV (fp16)", f64(dqkv), np.stack(b["dQKV"]))
    assert_close("dX", f64(dX), b["dXn"])
    assert_close("dW_qkv (packed)", f64(dWqkv), O.pack_qkv_weight(b["dW_qkv"], nh, dh, t))
    assert_close("db_qkv (packed)", f64(dbqkv), O.pack_qkv_bias(b["db_qkv"], nh, dh, t))
    assert_close("dW_o (packed)", f64(dWo), O.pack_row_weight(b["dW_o"], t))
    assert_close("db_o", f64(dbo), b["db_o"])
