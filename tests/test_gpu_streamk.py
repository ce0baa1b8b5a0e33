"""Split K across CTA pairs, against the fp64 oracle through the C ABI.

With a workspace, the tiles past the pair kernel's last full round of whole tiles (all
tiles, when there are fewer tiles than CTA pairs) may be cut into S equal K ranges at the
same k-stages, dealt to every pair, when the plan's time model says it pays (long K, few
tiles).  bf16-output GEMMs chain their ranges: range 0 stores its fp32 partial into the
tile's running sum in the workspace, each next range adds into it in L2 after the previous
range's flag, and the last range adds its accumulator and applies the epilogue.  The other
epilogues (and bf16 with TP_SPLIT_CHAIN=0) count their ranges: each range leaves its fp32
partial in the workspace and counts itself; the range that completes a tile's count adds
the partials in range order and applies the epilogue.
Covered here: the row-parallel GEMM with its fused shard sum (ranges that cross shard
boundaries, ragged M, N and K; a split past a full round of whole tiles; both forms), the
column-parallel GEMM with each activation, the backward's dgrad (with the fused
bias-gradient partials), both wgrads and the f-reduced dX, a workspace that holds only a
few partials or running sums,
determinism, CUDA-graph replay with new inputs between replays (the counters and flags
reset themselves), and guard bytes around the workspace (which starts with arbitrary
bytes) and every output.
Criterion: max|gpu - oracle| <= 1e-2 * max|oracle| per output.
"""

import numpy as np
import pytest
import torch

import oracle as O
from megatron_tensor_transformer_shard_gb300 import _lib as L
from megatron_tensor_transformer_shard_gb300 import inputs as I
from megatron_tensor_transformer_shard_gb300 import tp as T

from gpu_helpers import Guarded, assert_close, f64, guarded_ws

pytestmark = pytest.mark.gpu

SK_BYTES = 256 * (256 * 256 * 4 + 64)


def _case(M, h, F, t, seed, bias=True):
    inp = I.mlp_inputs(M, h, F, bias=bias, dy=True, seed=seed)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    ref = {k: (f64(v) if v is not None else None) for k, v in inp.items()}
    return dev, ref, T.MLPWeights(dev["W_up"], dev["b_up"], dev["W_down"], dev["b_down"], t)


@pytest.mark.parametrize("chain", [True, False])
@pytest.mark.parametrize("M,h,F,t", [
    (1000, 1024, 16384, 4),  # 16 tiles, 128 k-stages
    (520, 1032, 15680, 4),   # ragged M (3 row tiles), N (1032 = 4 x 256 + 8), K (3920 per shard)
    (300, 1024, 16384, 4),   # 8 tiles, 128 k-stages
    (272, 776, 24576, 3),    # 8 tiles, t = 3: range boundaries inside shards
    (2048, 4096, 12288, 4),  # 128 tiles: a round of whole tiles, then 52 kept whole (a split would not pay)
    (2560, 2048, 4096, 4),   # 80 tiles: a round of whole tiles, then the last few split
])
def test_row_parallel_streamk_matches_oracle(M, h, F, t, chain, monkeypatch):
    monkeypatch.setenv("TP_SPLIT_CHAIN", "1" if chain else "0")
    dev, ref, w = _case(M, h, F, t, seed=60 + t)
    A = (torch.randn(t, M, F // t, generator=torch.Generator().manual_seed(61)) * 0.5).to(torch.bfloat16)
    R = torch.randn(M, h, generator=torch.Generator().manual_seed(62)).to(torch.bfloat16)
    nws = L.tp_row_parallel_workspace_size(M, F, h, t)
    assert nws == SK_BYTES
    ws = guarded_ws(nws)
    Y = Guarded((M, h), torch.bfloat16)
    L.tp_row_parallel_forward_ws(A.cuda(), M, F, h, t, w.Wdown_p, dev["b_down"], R.cuda(), Y.t, ws.t, nws)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    ws.check("workspace")
    Y.check("Y")
    Af, Wd = f64(A), ref["W_down"]
    Ft = F // t
    ref_Y = sum(Af[i] @ Wd[i * Ft:(i + 1) * Ft] for i in range(t)) + ref["b_down"] + f64(R)
    assert_close("Y", f64(Y.t), ref_Y)
    # the data-parallel schedule (no workspace) agrees within the bound
    Y0 = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    L.tp_row_parallel_forward(A.cuda(), M, F, h, t, w.Wdown_p, dev["b_down"], R.cuda(), Y0)
    assert_close("stream-K vs data-parallel", f64(Y.t), f64(Y0))


@pytest.mark.parametrize("act", ["identity", "relu", "gelu_tanh", "gelu_erf"])
def test_column_parallel_streamk_activations(act):
    M, h, F, t = 600, 8200, 1024, 2       # 3 x 2 x 2 = 12 tiles, 129 k-blocks (ragged K): 4 ranges
    dev, ref, w = _case(M, h, F, t, seed=63)
    nws = L.tp_column_parallel_workspace_size(M, h, F, t)
    ws = guarded_ws(nws)
    Z, A = Guarded((t, M, F // t), torch.bfloat16), Guarded((t, M, F // t), torch.bfloat16)
    L.tp_column_parallel_forward_ws(dev["X"], M, h, F, t, L.ACT_BY_NAME[act], w.Wup_p, w.b_up, Z.t, A.t, ws.t, nws)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    for name, g in (("workspace", ws), ("Z", Z), ("A", A)):
        g.check(name)
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], ref["b_up"], ref["W_down"], ref["b_down"], act, t)
    assert_close("Z", f64(Z.t), np.stack(o["Z"]))
    assert_close("A", f64(A.t), np.stack(o["A"]))


@pytest.mark.parametrize("M,h,F,t", [(1000, 1024, 16384, 4),  # dX split
                                     (400, 4096, 1024, 2),    # dgrad * act' (and its db_up partials) split
                                     (16384, 512, 1024, 2)])  # both weight gradients split
def test_mlp_backward_streamk(M, h, F, t):
    """dgrad * act' with the fused db_up partials, both weight gradients and the f-reduced
    dX, with K split across CTA pairs where their tiles are few."""
    dev, ref, w = _case(M, h, F, t, seed=64)
    Y, Z, A = T.mlp_forward(dev["X"], w, "gelu_tanh")
    nws = L.tp_mlp_backward_workspace_size(M, h, F, t, 0)
    ws = guarded_ws(nws)
    out = {"dX": Guarded((M, h), torch.bfloat16), "dWup_p": Guarded((t, F // t, h), torch.float32),
           "dWdown_p": Guarded((t, h, F // t), torch.float32), "dbup": Guarded((F,), torch.float32),
           "dbdown": Guarded((h,), torch.float32)}
    L.tp_mlp_backward(dev["dY"], dev["X"], Z, A, M, h, F, t, L.TP_ACT_GELU_TANH, w.Wup_p, w.Wdown_p,
                      out["dX"].t, out["dWup_p"].t, out["dWdown_p"].t, out["dbup"].t, out["dbdown"].t, 0, 0,
                      ws.t, nws)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    ws.check("workspace")
    for k, g in out.items():
        g.check(k)
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], ref["b_up"], ref["W_down"], ref["b_down"], "gelu_tanh", t)
    b = O.mlp_backward_sharded(ref["dY"], ref["X"], ref["W_up"], ref["W_down"], o, "gelu_tanh", t)
    assert_close("dX", f64(out["dX"].t), b["dX"])
    assert_close("dW_up (packed)", f64(out["dWup_p"].t), O.pack_col_weight(b["dW_up"], t))
    assert_close("dW_down (packed)", f64(out["dWdown_p"].t), O.pack_row_weight(b["dW_down"], t))
    assert_close("db_up", f64(out["dbup"].t), b["db_up"])
    assert_close("db_down", f64(out["dbdown"].t), b["db_down"])


@pytest.mark.parametrize("slots", [2, 32, 48])
def test_partial_workspace_limits_the_clusters(slots):
    """A workspace with room for only a few partials or running sums (16 tiles: chained
    ranges need one running sum per tile, so 2 slots keep the tiles whole) still gives the
    result."""
    M, h, F, t = 1000, 1024, 16384, 4
    dev, ref, w = _case(M, h, F, t, seed=65)
    A = (torch.randn(t, M, F // t, generator=torch.Generator().manual_seed(66)) * 0.5).to(torch.bfloat16).cuda()
    nws = slots * (256 * 256 * 4 + 64)
    ws = guarded_ws(nws)
    Y = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    L.tp_row_parallel_forward_ws(A, M, F, h, t, w.Wdown_p, dev["b_down"], None, Y, ws.t, nws)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    ws.check("workspace")
    Af, Wd, Ft = f64(A.cpu()), ref["W_down"], F // t
    assert_close("Y", f64(Y), sum(Af[i] @ Wd[i * Ft:(i + 1) * Ft] for i in range(t)) + ref["b_down"])


def test_streamk_deterministic_and_graph_replay_with_new_inputs():
    """Same inputs, same bits; captured in a CUDA graph, each replay (with new inputs
    written between replays) gives the eager result for those inputs -- every replay
    repeats the flags' launch tag, and the flags start from zero because the last range of
    a tile resets them."""
    M, h, F, t = 1000, 1024, 16384, 4
    dev, ref, w = _case(M, h, F, t, seed=67)
    nws = L.tp_row_parallel_workspace_size(M, F, h, t)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    A = torch.empty(t, M, F // t, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    run = lambda: L.tp_row_parallel_forward_ws(A, M, F, h, t, w.Wdown_p, dev["b_down"], None, Y, ws, nws)
    inputs = [(torch.randn(t, M, F // t, generator=torch.Generator().manual_seed(70 + k)) * 0.5).to(torch.bfloat16)
              for k in range(3)]
    eager = []
    for x in inputs:
        A.copy_(x)
        outs = []
        for _ in range(2):
            run()
            torch.cuda.synchronize()
            outs.append(Y.clone())
        assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
        eager.append(outs[0])
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            run()
    torch.cuda.current_stream().wait_stream(cs)
    for rep in range(2):
        for x, ref_y in zip(inputs, eager):
            A.copy_(x)
            Y.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(Y.view(torch.int16), ref_y.view(torch.int16)), rep
    assert L.tp_get_device_status(check=False) == L.TP_OK
