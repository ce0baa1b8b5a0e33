"""GPU parity of the row-parallel GEMM with the g all-reduce overlapped tile by
tile (the explicit per-shard partials reduced while later tiles compute): the
exchanged partials match the oracle's per-shard products, Y matches the oracle,
and Y is bit-identical to the path that reduces the same partials afterwards.
Shapes cover tiles that one CTA pair walks shard after shard (more tiles than
pairs, more rounds than one), ragged M and h, t = 1..8 (not only powers of two),
a workspace of arbitrary contents, and CUDA-graph replay."""

import numpy as np
import pytest
import torch

import oracle as O
from megatron_tensor_transformer_shard_gb300 import _lib as L
from megatron_tensor_transformer_shard_gb300 import inputs as I

from gpu_helpers import assert_close, f64

pytestmark = pytest.mark.gpu


def _mlp(M, h, F, t, seed, residual=False):
    inp = I.mlp_inputs(M, h, F, bias=True, dy=False, seed=seed)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    Wup = torch.empty(t, F // t, h, dtype=torch.bfloat16, device="cuda")
    Wdn = torch.empty(t, h, F // t, dtype=torch.bfloat16, device="cuda")
    L.tp_pack_col(dev["W_up"], h, F, t, Wup)
    L.tp_pack_row(dev["W_down"], F, h, t, Wdn)
    res = torch.randn(M, h, generator=torch.Generator().manual_seed(seed + 1)).to(torch.bfloat16).cuda() if residual else None
    outs = {}
    for name, flag in (("fused", 0), ("unfused", L.TP_FLAG_UNFUSED_REDUCE), ("overlap", L.TP_FLAG_OVERLAP_REDUCE)):
        Y = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
        A = torch.empty(t, M, F // t, dtype=torch.bfloat16, device="cuda")
        nws = L.tp_mlp_workspace_size(M, h, F, t, flag)
        ws = torch.empty(max(nws, 256), dtype=torch.uint8, device="cuda")
        L.tp_mlp_forward(dev["X"], M, h, F, t, L.ACT_BY_NAME["gelu_tanh"], Wup, dev["b_up"], Wdn, dev["b_down"], res,
                         Y, None, A, flag, ws, ws.numel())
        outs[name] = (Y, A)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    return inp, dev, Wdn, res, outs


@pytest.mark.parametrize("M,h,F,t", [(300, 512, 1024, 2), (512, 264, 2048, 4), (384, 256, 4096, 8),
                                     (2304, 2312, 1536, 4),   # 9 x 10 tiles: two rounds of CTA pairs
                                     (4100, 4096, 768, 3),    # 17 x 16 tiles, t = 3, ragged M
                                     (520, 1024, 1024, 1)])
def test_overlap_matches_oracle_and_unfused_bits(M, h, F, t):
    inp, dev, Wdn, res, outs = _mlp(M, h, F, t, seed=M + t, residual=(t == 4))
    ref = {k: (f64(v) if v is not None else None) for k, v in inp.items()}
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], ref["b_up"], ref["W_down"], ref["b_down"], "gelu_tanh", t)
    want = o["Y"] + (f64(res) if res is not None else 0.0)
    assert_close("Y overlap", f64(outs["overlap"][0]), want)
    # same partials, same order of additions: the same bits as the reduction run afterwards
    assert torch.equal(outs["overlap"][0].view(torch.int16), outs["unfused"][0].view(torch.int16))


def test_overlap_partials_are_the_shard_products():
    M, h, F, t = 300, 256, 1024, 4
    inp, dev, Wdn, res, outs = _mlp(M, h, F, t, seed=5)
    A = outs["overlap"][1]
    P = torch.empty(t, M, h, dtype=torch.float32, device="cuda")
    Y = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    nws = L.tp_row_parallel_overlap_workspace_size(M, F, h, t)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    L.tp_row_parallel_forward_overlap(A, M, F, h, t, Wdn, dev["b_down"], None, Y, P, ws, nws)
    torch.cuda.synchronize()
    A64, W64 = f64(A), f64(inp["W_down"])
    Ft = F // t
    for i in range(t):
        assert_close(f"P[{i}]", f64(P[i]), A64[i] @ W64[i * Ft:(i + 1) * Ft])
    assert torch.equal(Y.view(torch.int16), outs["overlap"][0].view(torch.int16))


def test_overlap_rejects_small_or_wide():
    x = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    assert L.tp_row_parallel_forward_overlap(x, 128, 64, 64, 2, x, None, None, x, None, ws, ws.numel(),
                                             check=False) == L.TP_ERR_UNSUPPORTED      # M <= 128
    assert L.tp_row_parallel_forward_overlap(x, 256, 144, 64, 9, x, None, None, x, None, ws, ws.numel(),
                                             check=False) == L.TP_ERR_SHAPE            # t > 8
    assert L.tp_row_parallel_forward_overlap(x, 256, 64, 64, 2, x, None, None, x, None, ws, 16,
                                             check=False) == L.TP_ERR_WORKSPACE


def test_overlap_graph_replay_with_new_inputs_and_garbage_workspace():
    """The running sums need no initial contents: eager runs on a workspace filled with
    0xff match the fp32 sum of the shard products, and CUDA-graph replays with new inputs
    written between them give the eager bits."""
    M, h, F, t = 2304, 2312, 1536, 4
    Ft = F // t
    gen = torch.Generator().manual_seed(90)
    W = (torch.randn(t, h, Ft, generator=gen) * 0.05).to(torch.bfloat16).cuda()
    bias = torch.randn(h, generator=gen).to(torch.bfloat16).cuda()
    inputs = [(torch.randn(t, M, Ft, generator=gen) * 0.5).to(torch.bfloat16) for _ in range(3)]
    A = torch.empty(t, M, Ft, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    nws = L.tp_row_parallel_overlap_workspace_size(M, F, h, t)
    ws = torch.full((nws,), 255, dtype=torch.uint8, device="cuda")
    run = lambda: L.tp_row_parallel_forward_overlap(A, M, F, h, t, W, bias, None, Y, None, ws, nws)
    want = []
    for x in inputs:
        A.copy_(x)
        P = torch.stack([A[i].float() @ W[i].float().t() for i in range(t)])
        run()
        torch.cuda.synchronize()
        want.append(Y.clone())
        assert_close("Y", f64(Y), f64(P.sum(0) + bias.float()))
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            run()
    torch.cuda.current_stream().wait_stream(cs)
    for rep in range(2):
        for x, ref_y in zip(inputs, want):
            A.copy_(x)
            Y.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(Y.view(torch.int16), ref_y.view(torch.int16)), rep
    assert L.tp_get_device_status(check=False) == L.TP_OK


@pytest.mark.slow
def test_overlap_full_size_c2():
    c = I.CONFIGS["c2"]
    inp, dev, Wdn, res, outs = _mlp(c["M"], c["h"], c["F"], c["t"], seed=0)
    assert torch.equal(outs["overlap"][0].view(torch.int16), outs["unfused"][0].view(torch.int16))
    d = (outs["overlap"][0].float() - outs["fused"][0].float()).abs().max().item()
    assert d <= 1e-2 * outs["fused"][0].float().abs().max().item()
