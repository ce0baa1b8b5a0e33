"""Split K for GEMMs with too few output tiles to occupy the GPU (M <= 128 tokens:
one 128-row tile), against the fp64 oracle through the C ABI.

The S CTAs of a thread-block cluster compute one output tile, each over one range of
its K steps -- for the row-parallel GEMM the t shards' K ranges laid end to end -- and
sum their fp32 partials through distributed shared memory in range order before the
epilogue (bias, activation, residual).  TP_SPLITK sets S (a power of two up to 16) so
that ragged ranges (S not dividing the k-steps, ranges that cross a shard boundary, K
not a multiple of the 64-deep k-block) are exercised; TP_SPLITC_NARROW picks 128- or
256-column tiles (N ragged against either).  Criterion as everywhere:
max|gpu - oracle| <= 1e-2 * max|oracle| per output, and the outputs sit between guard
bytes that must come back unchanged.
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


def _case(M, h, F, t, seed, bias=True):
    inp = I.mlp_inputs(M, h, F, bias=bias, dy=True, seed=seed)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    ref = {k: (f64(v) if v is not None else None) for k, v in inp.items()}
    return dev, ref, T.MLPWeights(dev["W_up"], dev["b_up"], dev["W_down"], dev["b_down"], t)


def _forward_guarded(dev, w, M, h, F, t, act, residual=None):
    # the split needs no scratch: no workspace is passed
    Y, Z, A = Guarded((M, h), torch.bfloat16), Guarded((t, M, F // t), torch.bfloat16), \
        Guarded((t, M, F // t), torch.bfloat16)
    L.tp_mlp_forward(dev["X"], M, h, F, t, L.ACT_BY_NAME[act], w.Wup_p, w.b_up, w.Wdown_p, w.b_down, residual,
                     Y.t, Z.t, A.t, 0, None, 0)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    for name, g in (("Y", Y), ("Z", Z), ("A", A)):
        g.check(name)
    return Y.t, Z.t, A.t


@pytest.mark.parametrize("narrow", ["0", "1"])
@pytest.mark.parametrize("S", ["", "2", "4", "8", "16"])
@pytest.mark.parametrize("M,h,F,t", [(128, 1024, 4096, 2), (100, 392, 1296, 2), (37, 264, 3072, 4)])
def test_split_forward_matches_oracle(M, h, F, t, S, narrow, monkeypatch):
    """h = 392 and 264 are not multiples of 64 (the last k-block is ragged); F/t = 648
    gives 11 k-blocks per shard, so the row-parallel GEMM's 22 k-steps cut into 4 or 8
    ranges put a boundary inside a shard's K range; 16 ranges of the column GEMM's 7
    k-steps are capped at 4 (a power of two no larger than the k-steps)."""
    monkeypatch.setenv("TP_SPLITK", S)
    monkeypatch.setenv("TP_SPLITC_NARROW", narrow)
    dev, ref, w = _case(M, h, F, t, seed=30 + M)
    Y, Z, A = _forward_guarded(dev, w, M, h, F, t, "gelu_tanh")
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], ref["b_up"], ref["W_down"], ref["b_down"], "gelu_tanh", t)
    assert_close("Z", f64(Z), np.stack(o["Z"]))
    assert_close("A", f64(A), np.stack(o["A"]))
    assert_close("Y", f64(Y), o["Y"])


@pytest.mark.parametrize("act", ["identity", "relu", "gelu_erf"])
def test_split_forward_activations_and_residual(act, monkeypatch):
    monkeypatch.setenv("TP_SPLITK", "4")
    M, h, F, t = 96, 512, 2048, 4
    dev, ref, w = _case(M, h, F, t, seed=41)
    R = torch.randn(M, h, generator=torch.Generator().manual_seed(42)).to(torch.bfloat16)
    Y, Z, A = _forward_guarded(dev, w, M, h, F, t, act, residual=R.cuda())
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], ref["b_up"], ref["W_down"], ref["b_down"], act, t)
    assert_close("A", f64(A), np.stack(o["A"]))
    assert_close("Y", f64(Y), o["Y"] + f64(R))


def test_split_bias_added_once(monkeypatch):
    """Zero weights: every K range's partial is zero; the epilogue adds b_down once."""
    monkeypatch.setenv("TP_SPLITK", "4")
    M, h, F, t = 64, 256, 2048, 4
    X = torch.randn(M, h).to(torch.bfloat16).cuda()
    w = T.MLPWeights(torch.zeros(h, F, dtype=torch.bfloat16, device="cuda"),
                     torch.zeros(F, dtype=torch.bfloat16, device="cuda"),
                     torch.zeros(F, h, dtype=torch.bfloat16, device="cuda"), torch.randn(h).to(torch.bfloat16).cuda(),
                     t)
    Y, _, _ = T.mlp_forward(X, w, "gelu_tanh")
    assert torch.equal(Y, w.b_down.expand(M, h))


def test_split_is_deterministic_and_close_to_unsplit(monkeypatch):
    """Same inputs, same bits on every call; against the unsplit GEMM only the rounding of
    the fp32 sum differs."""
    M, h, F, t = 128, 1024, 4096, 2
    dev, ref, w = _case(M, h, F, t, seed=43)
    runs = [T.mlp_forward(dev["X"], w, "gelu_tanh")[0].clone() for _ in range(3)]
    assert all(torch.equal(r.view(torch.int16), runs[0].view(torch.int16)) for r in runs[1:])
    monkeypatch.setenv("TP_SPLITK", "1")
    Y1, _, _ = T.mlp_forward(dev["X"], w, "gelu_tanh")
    assert_close("split vs unsplit", f64(runs[0]), f64(Y1))


@pytest.mark.parametrize("S", ["", "8"])
def test_split_backward_dx(S, monkeypatch):
    """The backward's f-reduced dX GEMM (t shards' K ranges end to end) splits at M <= 128."""
    monkeypatch.setenv("TP_SPLITK", S)
    M, h, F, t = 80, 264, 1296, 2
    dev, ref, w = _case(M, h, F, t, seed=44)
    Y, Z, A = T.mlp_forward(dev["X"], w, "gelu_tanh")
    nws = L.tp_mlp_backward_workspace_size(M, h, F, t, 0)
    ws = guarded_ws(nws)
    dX = Guarded((M, h), torch.bfloat16)
    g = {k: torch.empty(*s, dtype=torch.float32, device="cuda") for k, s in
         (("dWup_p", (t, F // t, h)), ("dWdown_p", (t, h, F // t)), ("dbup", (F,)), ("dbdown", (h,)))}
    L.tp_mlp_backward(dev["dY"], dev["X"], Z, A, M, h, F, t, L.TP_ACT_GELU_TANH, w.Wup_p, w.Wdown_p, dX.t,
                      g["dWup_p"], g["dWdown_p"], g["dbup"], g["dbdown"], 0, 0, ws.t, nws)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    ws.check("workspace")
    dX.check("dX")
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], ref["b_up"], ref["W_down"], ref["b_down"], "gelu_tanh", t)
    b = O.mlp_backward_sharded(ref["dY"], ref["X"], ref["W_up"], ref["W_down"], o, "gelu_tanh", t)
    assert_close("dX", f64(dX.t), b["dX"])
    assert_close("dW_up (packed)", f64(g["dWup_p"]), O.pack_col_weight(b["dW_up"], t))
    assert_close("db_up", f64(g["dbup"]), b["db_up"])


@pytest.mark.parametrize("S", ["", "16"])
def test_standalone_entry_points(S, monkeypatch):
    """tp_column_parallel_forward / tp_row_parallel_forward split K by themselves at M <= 128
    (no workspace): the oracle's results, and, for the output bias and residual, the same
    results as the unsplit GEMM within the bound."""
    monkeypatch.setenv("TP_SPLITK", S)
    M, h, F, t = 128, 1024, 4096, 2
    dev, ref, w = _case(M, h, F, t, seed=45)
    act = L.ACT_BY_NAME["gelu_tanh"]
    R = torch.randn(M, h, generator=torch.Generator().manual_seed(46)).to(torch.bfloat16).cuda()
    A = Guarded((t, M, F // t), torch.bfloat16)
    Y = Guarded((M, h), torch.bfloat16)
    L.tp_column_parallel_forward(dev["X"], M, h, F, t, act, w.Wup_p, w.b_up, None, A.t)
    L.tp_row_parallel_forward(A.t, M, F, h, t, w.Wdown_p, w.b_down, R, Y.t)
    A.check("A")
    Y.check("Y")
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], ref["b_up"], ref["W_down"], ref["b_down"], "gelu_tanh", t)
    assert_close("A", f64(A.t), np.stack(o["A"]))
    assert_close("Y", f64(Y.t), o["Y"] + f64(R))
    monkeypatch.setenv("TP_SPLITK", "1")
    Y1 = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    L.tp_row_parallel_forward(A.t, M, F, h, t, w.Wdown_p, w.b_down, R, Y1)
    assert_close("split vs unsplit", f64(Y.t), f64(Y1))


def test_split_graph_replay_matches_eager():
    """The split forward captured in a CUDA graph and replayed gives the eager call's bits."""
    M, h, F, t = 128, 1024, 4096, 2
    dev, ref, w = _case(M, h, F, t, seed=47)
    act = L.ACT_BY_NAME["gelu_tanh"]
    Y = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    A = torch.empty(t, M, F // t, dtype=torch.bfloat16, device="cuda")
    fwd = lambda: L.tp_mlp_forward(dev["X"], M, h, F, t, act, w.Wup_p, w.b_up, w.Wdown_p, w.b_down, None, Y, None,
                                   A, 0, None, 0)
    fwd()
    torch.cuda.synchronize()
    Y0 = Y.clone()
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            fwd()
    torch.cuda.current_stream().wait_stream(cs)
    for _ in range(3):
        Y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(Y.view(torch.int16), Y0.view(torch.int16))
