"""GPU parity of the TP MLP (packing, forward, backward) against the fp64
oracle, through the C ABI.

Criterion: bit-exact for packing; max|gpu - oracle| <= 1e-2 * max|oracle| per
floating-point output tensor.  Sizes span several 128x256 output tiles with
ragged tails in M, N and K (and the full-size workloads on sampled outputs).
"""

import numpy as np
import pytest
import torch

import oracle as O
from megatron_tensor_transformer_shard_gb300 import _lib as L
from megatron_tensor_transformer_shard_gb300 import inputs as I
from megatron_tensor_transformer_shard_gb300 import tp as T

from gpu_helpers import Guarded, assert_close, f64, guarded_ws, ws_bytes

pytestmark = pytest.mark.gpu


def _rand_bits(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 65536, shape, generator=g, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)


# ---------------------------------------------------------------- packing

@pytest.mark.parametrize("h,F,t", [(64, 256, 4), (40, 48, 2), (1024, 4096, 2), (136, 1024, 8)])
def test_pack_col_row_bit_exact(h, F, t):
    W = _rand_bits((h, F), 1)
    Wd = _rand_bits((F, h), 2)
    Wp = torch.empty(t, F // t, h, dtype=torch.bfloat16, device="cuda")
    Wdp = torch.empty(t, h, F // t, dtype=torch.bfloat16, device="cuda")
    L.tp_pack_col(W.cuda(), h, F, t, Wp)
    L.tp_pack_row(Wd.cuda(), F, h, t, Wdp)
    assert np.array_equal(I.bits(Wp.cpu()), O.pack_col_weight(I.bits(W), t))
    assert np.array_equal(I.bits(Wdp.cpu()), O.pack_row_weight(I.bits(Wd), t))
    back = torch.empty(h, F, dtype=torch.bfloat16, device="cuda")
    L.tp_unpack_col(Wp, h, F, t, back)
    assert np.array_equal(I.bits(back.cpu()), I.bits(W))
    backd = torch.empty(F, h, dtype=torch.bfloat16, device="cuda")
    L.tp_unpack_row(Wdp, F, h, t, backd)
    assert np.array_equal(I.bits(backd.cpu()), I.bits(Wd))


def test_pack_reshard_t_to_t_prime():
    h, F = 128, 1024
    W = _rand_bits((h, F), 3).cuda()
    p4 = torch.empty(4, F // 4, h, dtype=torch.bfloat16, device="cuda")
    L.tp_pack_col(W, h, F, 4, p4)
    un = torch.empty(h, F, dtype=torch.bfloat16, device="cuda")
    L.tp_unpack_col(p4, h, F, 4, un)
    p8 = torch.empty(8, F // 8, h, dtype=torch.bfloat16, device="cuda")
    L.tp_pack_col(un, h, F, 8, p8)
    assert np.array_equal(I.bits(p8.cpu()), O.pack_col_weight(I.bits(W.cpu()), 8))


@pytest.mark.parametrize("h,F,t", [(64, 512, 2), (96, 1024, 4)])
def test_pack_swiglu_bit_exact(h, F, t):
    Wg, Wu = _rand_bits((h, F), 4), _rand_bits((h, F), 5)
    out = torch.empty(2 * F, h, dtype=torch.bfloat16, device="cuda")
    L.tp_pack_swiglu(Wg.cuda(), Wu.cuda(), h, F, t, out)
    ref = O.pack_swiglu_weight(I.bits(Wg), I.bits(Wu), t, 128).reshape(2 * F, h)
    assert np.array_equal(I.bits(out.cpu()), ref)


@pytest.mark.parametrize("nh,dh,t", [(4, 16, 2), (8, 128, 8), (6, 64, 3)])
def test_pack_qkv_bit_exact(nh, dh, t):
    d = nh * dh
    W = _rand_bits((d, 3 * d), 6)
    b = _rand_bits((3 * d,), 7)
    Wp = torch.empty(t, 3 * d // t, d, dtype=torch.bfloat16, device="cuda")
    bp = torch.empty(t, 3 * d // t, dtype=torch.bfloat16, device="cuda")
    L.tp_pack_qkv_heads(W.cuda(), d, nh, dh, t, Wp)
    L.tp_pack_qkv_bias(b.cuda(), d, nh, dh, t, bp)
    assert np.array_equal(I.bits(Wp.cpu()), O.pack_qkv_weight(I.bits(W), nh, dh, t))
    assert np.array_equal(I.bits(bp.cpu()), O.pack_qkv_bias(I.bits(b), nh, dh, t))
    back = torch.empty(d, 3 * d, dtype=torch.bfloat16, device="cuda")
    L.tp_unpack_qkv_heads(Wp, d, nh, dh, t, back)
    assert np.array_equal(I.bits(back.cpu()), I.bits(W))


# ---------------------------------------------------------------- MLP

def _case(M, h, F, t, seed=0, bias=True):
    inp = I.mlp_inputs(M, h, F, bias=bias, dy=True, seed=seed)
    dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    ref = {k: (f64(v) if v is not None else None) for k, v in inp.items()}
    w = T.MLPWeights(dev["W_up"], dev["b_up"], dev["W_down"], dev["b_down"], t)
    return dev, ref, w


SHAPES = [
    (128, 1024, 4096, 2),   # the forward-only workload, full size
    (200, 264, 784, 2),     # ragged M, N (F/t = 392) and K (h = 264)
    (1, 64, 128, 4),        # a single token
    (300, 512, 2048, 8),
    (257, 128, 1536, 4),
]


@pytest.mark.parametrize("M,h,F,t", SHAPES)
def test_mlp_forward_parity(M, h, F, t):
    dev, ref, w = _case(M, h, F, t)
    Y, Z, A = T.mlp_forward(dev["X"], w, "gelu_tanh")
    torch.cuda.synchronize()
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], ref["b_up"], ref["W_down"], ref["b_down"], "gelu_tanh", t)
    assert_close("Y", f64(Y), o["Y"])
    assert_close("Z", f64(Z), np.stack(o["Z"]))
    assert_close("A", f64(A), np.stack(o["A"]))
    assert L.tp_get_device_status(check=False) == L.TP_OK


@pytest.mark.parametrize("act", ["identity", "relu", "gelu_tanh", "gelu_erf"])
def test_mlp_forward_activations(act):
    M, h, F, t = 192, 256, 1024, 4
    dev, ref, w = _case(M, h, F, t, seed=1)
    Y, Z, A = T.mlp_forward(dev["X"], w, act)
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], ref["b_up"], ref["W_down"], ref["b_down"], act, t)
    assert_close("Y", f64(Y), o["Y"])
    assert_close("A", f64(A), np.stack(o["A"]))


def test_mlp_forward_residual_and_no_bias():
    M, h, F, t = 130, 256, 512, 2
    dev, ref, w = _case(M, h, F, t, seed=2, bias=False)
    R = torch.randn(M, h, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    Y, _, _ = T.mlp_forward(dev["X"], w, "gelu_tanh", residual=R.cuda(), save_z=False)
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], None, ref["W_down"], None, "gelu_tanh", t)
    assert_close("Y", f64(Y), o["Y"] + f64(R))


@pytest.mark.parametrize("M,h,F,t", [(200, 264, 784, 2), (256, 512, 2048, 4)])
def test_unfused_partials_match_oracle(M, h, F, t):
    """TP_FLAG_UNFUSED_REDUCE writes each shard's partial P_i; check every P_i
    and the reduced output against the oracle, and against the fused path."""
    dev, ref, w = _case(M, h, F, t, seed=3)
    flags = L.TP_FLAG_UNFUSED_REDUCE
    nws = L.tp_mlp_workspace_size(M, h, F, t, flags)
    assert nws >= t * M * h * 4                     # the partials first, then the split-K room
    wsb = torch.empty(nws, dtype=torch.uint8, device="cuda")
    ws = wsb[:t * M * h * 4].view(torch.float32).view(t, M, h)
    Y = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    A = torch.empty(t, M, F // t, dtype=torch.bfloat16, device="cuda")
    L.tp_mlp_forward(dev["X"], M, h, F, t, L.TP_ACT_GELU_TANH, w.Wup_p, w.b_up, w.Wdown_p, w.b_down, None, Y,
                     None, A, flags, wsb, nws)
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], ref["b_up"], ref["W_down"], ref["b_down"], "gelu_tanh", t)
    for i in range(t):
        assert_close(f"P_{i}", f64(ws[i]), o["P"][i])
    assert_close("Y", f64(Y), o["Y"])
    Yf, _, _ = T.mlp_forward(dev["X"], w, "gelu_tanh")
    assert_close("fused vs unfused", f64(Yf), f64(Y))


def test_bias_added_once_on_gpu():
    """Zero weights: Y must equal b_down exactly once (not t times)."""
    M, h, F, t = 64, 128, 512, 4
    X = torch.randn(M, h).to(torch.bfloat16).cuda()
    Wu = torch.zeros(h, F, dtype=torch.bfloat16, device="cuda")
    Wd = torch.zeros(F, h, dtype=torch.bfloat16, device="cuda")
    bu = torch.zeros(F, dtype=torch.bfloat16, device="cuda")
    bd = torch.randn(h).to(torch.bfloat16).cuda()
    w = T.MLPWeights(Wu, bu, Wd, bd, t)
    for flags in (0, L.TP_FLAG_UNFUSED_REDUCE):
        Y, _, _ = T.mlp_forward(X, w, "gelu_tanh", flags=flags)
        assert torch.equal(Y, bd.expand(M, h)), flags


@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("M,h,F,t", [(384, 264, 784, 2), (1000, 512, 2048, 4)])
def test_single_cta_and_pair_gemm_paths(M, h, F, t, pair, monkeypatch):
    """Both GEMM kernels (one CTA per 128x256 tile, and CTA pairs per 256x256
    tile through tcgen05 cta_group::2) give the oracle's results, forward and
    backward (all four operand-major combinations)."""
    monkeypatch.setenv("TP_GEMM_PAIR", pair)
    _backward_check(M, h, F, t, "gelu_tanh", seed=8)


@pytest.mark.parametrize("pair", ["0", "1"])
def test_gemm_operand_copies_odd_k_blocks(pair, monkeypatch):
    """Operand tiles arrive in one 4-D TMA copy per stage where K (K-major) or the row count
    (MN-major) is a multiple of 64, and one-output GEMMs of the pair kernel take two 64-wide
    k-blocks per stage.  Here every K is a multiple of 64 with an odd number of k-blocks: h =
    192 (dgrad, 3 blocks), F/t = 320 (row-parallel and dX, 5 blocks per shard, summed over the
    shards), M = 320 tokens (wgrad, 5 blocks).  So each shard's last stage carries a second,
    out-of-range k-block that must arrive as zeros and not as the next shard's data."""
    monkeypatch.setenv("TP_GEMM_PAIR", pair)
    M, h, F, t = 320, 192, 640, 2
    dev, ref, w = _case(M, h, F, t, seed=12)
    Y, _, _ = T.mlp_forward(dev["X"], w, "gelu_tanh")
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], ref["b_up"], ref["W_down"], ref["b_down"], "gelu_tanh", t)
    assert_close("Y", f64(Y), o["Y"])
    _backward_check(M, h, F, t, "gelu_tanh", seed=12)


def test_mlp_zero_tokens():
    dev, ref, w = _case(8, 64, 256, 2)
    Y = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    A = torch.empty(2, 0, 128, dtype=torch.bfloat16, device="cuda")
    L.tp_mlp_forward(dev["X"], 0, 64, 256, 2, 2, w.Wup_p, w.b_up, w.Wdown_p, w.b_down, None, Y, None, A, 0, None, 0)


def _backward_check(M, h, F, t, act, seed, flags=0):
    dev, ref, w = _case(M, h, F, t, seed=seed)
    Y, Z, A = T.mlp_forward(dev["X"], w, act)
    g = T.mlp_backward(dev["dY"], dev["X"], Z, A, w, act, flags=flags)
    torch.cuda.synchronize()
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], ref["b_up"], ref["W_down"], ref["b_down"], act, t)
    b = O.mlp_backward_sharded(ref["dY"], ref["X"], ref["W_up"], ref["W_down"], o, act, t)
    assert_close("dX", f64(g["dX"]), b["dX"])
    assert_close("dW_up (packed)", f64(g["dWup_p"]), O.pack_col_weight(b["dW_up"], t))
    assert_close("dW_down (packed)", f64(g["dWdown_p"]), O.pack_row_weight(b["dW_down"], t))
    assert_close("db_up", f64(g["dbup"]), b["db_up"])
    assert_close("db_down", f64(g["dbdown"]), b["db_down"])
    return dev, w, g, (Y, Z, A)


@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("M", [1, 33, 64, 96, 161])
def test_backward_small_and_ragged_m_guarded(M, pair, monkeypatch):
    """db_up's per-32-row partials come from the dgrad epilogue.  When the last row tile
    has 32-row blocks wholly past M (M <= 96 on the single-CTA kernel, or M % 128 in
    1..96 with TP_GEMM_PAIR=0), those blocks must write nothing: not into the next
    shard's first block, not past the workspace.  The workspace and every output sit
    between guard bytes that must come back unchanged, and every gradient (db_up above
    all) must match the oracle."""
    monkeypatch.setenv("TP_GEMM_PAIR", pair)
    h, F, t = 128, 1024, 4
    dev, ref, w = _case(M, h, F, t, seed=21 + M)
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


@pytest.mark.parametrize("M,h,F,t", [(200, 264, 784, 2), (256, 512, 2048, 4), (130, 128, 1024, 8)])
def test_mlp_backward_parity(M, h, F, t):
    _backward_check(M, h, F, t, "gelu_tanh", seed=4)


@pytest.mark.parametrize("act", ["identity", "relu", "gelu_erf"])
def test_mlp_backward_activations(act):
    _backward_check(192, 256, 1024, 4, act, seed=5)


def test_mlp_backward_unfused_and_accumulate():
    M, h, F, t = 256, 256, 1024, 4
    dev, w, g, (Y, Z, A) = _backward_check(M, h, F, t, "gelu_tanh", seed=6, flags=L.TP_FLAG_UNFUSED_REDUCE)
    g2 = T.mlp_backward(dev["dY"], dev["X"], Z, A, w, "gelu_tanh")
    assert_close("fused dX vs unfused", f64(g2["dX"]), f64(g["dX"]))
    base = {k: g2[k].clone() for k in ("dWup_p", "dWdown_p", "dbup", "dbdown")}
    g3 = T.mlp_backward(dev["dY"], dev["X"], Z, A, w, "gelu_tanh", grads={k: v.clone() for k, v in base.items()})
    for k in base:
        assert_close(k + " accumulated", f64(g3[k]), 2 * f64(base[k]))


def test_autograd_function():
    M, h, F, t = 128, 256, 1024, 2
    dev, ref, w = _case(M, h, F, t, seed=7)
    X = dev["X"].clone().requires_grad_()
    Y = T.TPMLPFunction.apply(X, w, "gelu_tanh")
    Y.backward(dev["dY"])
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], ref["b_up"], ref["W_down"], ref["b_down"], "gelu_tanh", t)
    b = O.mlp_backward_sharded(ref["dY"], ref["X"], ref["W_up"], ref["W_down"], o, "gelu_tanh", t)
    assert_close("Y", f64(Y), o["Y"])
    assert_close("dX", f64(X.grad), b["dX"])
    assert_close("dW_up", f64(w.grads["dWup_p"]), O.pack_col_weight(b["dW_up"], t))


def test_first_call_from_a_new_thread():
    """A thread whose first CUDA work is a library call (the autograd worker
    thread does this) must get a current context before tensor maps are
    encoded; the GEMM must not fail with TP_ERR_CUDA there."""
    import threading
    M, h, F, t = 128, 256, 1024, 2
    dev, ref, w = _case(M, h, F, t, seed=12)
    Y, Z, A = T.mlp_forward(dev["X"], w, "gelu_tanh")
    torch.cuda.synchronize()
    box = {}

    def worker():
        try:
            box["g"] = T.mlp_backward(dev["dY"], dev["X"], Z, A, w, "gelu_tanh")
            torch.cuda.synchronize()
        except Exception as e:  # reported below
            box["err"] = e

    th = threading.Thread(target=worker)
    th.start()
    th.join()
    assert "err" not in box, box.get("err")
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], ref["b_up"], ref["W_down"], ref["b_down"], "gelu_tanh", t)
    b = O.mlp_backward_sharded(ref["dY"], ref["X"], ref["W_up"], ref["W_down"], o, "gelu_tanh", t)
    assert_close("dX", f64(box["g"]["dX"]), b["dX"])


# ------------------------------------------------ full-size workloads (sampled)

def _rows(M, n=12):
    return sorted(set([0, 1, 127, 128, M // 2, M - 129, M - 1] + list(np.random.default_rng(0).integers(0, M, n))))


@pytest.mark.slow
def test_full_size_fwd_bwd_sampled():
    """The 2048x4096 -> 16384, t = 4 forward+backward in the launch configuration
    the bench times; compared on sampled rows of Y and dX and sampled rows /
    columns of the weight gradients, each computed by the oracle one by one."""
    cfg = I.CONFIGS["c2"]
    M, h, F, t = cfg["M"], cfg["h"], cfg["F"], cfg["t"]
    inp = I.mlp_inputs(M, h, F, bias=True, dy=True, seed=0)
    dev = {k: v.cuda() for k, v in inp.items()}
    w = T.MLPWeights(dev["W_up"], dev["b_up"], dev["W_down"], dev["b_down"], t)
    Y, Z, A = T.mlp_forward(dev["X"], w, "gelu_tanh")
    g = T.mlp_backward(dev["dY"], dev["X"], Z, A, w, "gelu_tanh")
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    X, Wu, bu, Wd, bd, G = (f64(inp[k]) for k in ("X", "W_up", "b_up", "W_down", "b_down", "dY"))
    rows = _rows(M)
    o = O.mlp_forward_sharded(X[rows], Wu, bu, Wd, bd, "gelu_tanh", t)
    assert_close("Y rows", f64(Y[rows]), o["Y"])
    b = O.mlp_backward_sharded(G[rows], X[rows], Wu, Wd, o, "gelu_tanh", t)
    assert_close("dX rows", f64(g["dX"][rows]), b["dX"])
    # weight-gradient columns need every token: pick a few hidden units f
    fs = [0, 1, 255, 256, F // t - 1, F // t, F // 2 + 7, F - 1]
    Zc = X @ Wu[:, fs] + bu[fs]
    dZc = (G @ Wd[fs, :].T) * O.act_grad("gelu_tanh", Zc)
    dWu_cols = X.T @ dZc                               # dW_up[:, f]
    Ac = O.act("gelu_tanh", Zc)
    dWd_rows = Ac.T @ G                                # dW_down[f, :]
    Ft = F // t
    gu = g["dWup_p"].reshape(F, h)                     # packed [t][Ft][h] == dW_up^T
    gd = g["dWdown_p"].cpu()                           # [t][h][Ft]
    got_u = f64(gu[fs]).T
    got_d = np.stack([f64(gd[f // Ft, :, f % Ft]) for f in fs])
    assert_close("dW_up columns", got_u, dWu_cols)
    assert_close("dW_down rows", got_d, dWd_rows)
    assert_close("db_up sampled", f64(g["dbup"])[fs], dZc.sum(axis=0))
    assert_close("db_down", f64(g["dbdown"]), G.sum(axis=0))


# ---------------------------------------------------------------- failure paths

def test_bounded_wait_timeout_reported_and_context_survives():
    assert L.tp_get_device_status(check=False) == L.TP_OK
    L.tp_selftest_bounded_wait(20000)   # 20 ms
    assert L.tp_get_device_status(check=False) == L.TP_ERR_TIMEOUT
    assert L.tp_get_device_status(check=False) == L.TP_OK   # cleared
    dev, ref, w = _case(64, 128, 256, 2)
    Y, _, _ = T.mlp_forward(dev["X"], w, "gelu_tanh")
    o = O.mlp_forward_sharded(ref["X"], ref["W_up"], ref["b_up"], ref["W_down"], ref["b_down"], "gelu_tanh", 2)
    assert_close("Y after timeout", f64(Y), o["Y"])


def test_host_validation_on_device():
    dev, ref, w = _case(64, 128, 256, 2)
    Y = torch.empty(64, 128, dtype=torch.bfloat16, device="cuda")
    A = torch.empty(2, 64, 128, dtype=torch.bfloat16, device="cuda")
    base = dev["X"].data_ptr()
    r = L.tp_mlp_forward(base + 2, 64, 128, 256, 2, 2, w.Wup_p, w.b_up, w.Wdown_p, w.b_down, None, Y, None, A, 0,
                         None, 0, check=False)
    assert r == L.TP_ERR_ALIGN
    r = L.tp_mlp_forward(dev["X"], 64, 128, 256, 3, 2, w.Wup_p, w.b_up, w.Wdown_p, w.b_down, None, Y, None, A, 0,
                         None, 0, check=False)
    assert r == L.TP_ERR_SHAPE
    small = ws_bytes(16)
    r = L.tp_mlp_forward(dev["X"], 64, 128, 256, 2, 2, w.Wup_p, w.b_up, w.Wdown_p, w.b_down, None, Y, None, A,
                         L.TP_FLAG_UNFUSED_REDUCE, small, 16, check=False)
    assert r == L.TP_ERR_WORKSPACE


@pytest.mark.parametrize("M,h,F,t", [(128, 1024, 4096, 2), (512, 512, 2048, 4)])
def test_mlp_forward_graph_replay_matches_eager(M, h, F, t):
    """The forward's GEMMs launch with programmatic dependent launch; captured in a
    CUDA graph and replayed they give the same bits as the eager call."""
    inp = I.mlp_inputs(M, h, F, bias=True, dy=False, seed=13, device="cuda")
    w = T.MLPWeights(inp["W_up"], inp["b_up"], inp["W_down"], inp["b_down"], t)
    act = L.ACT_BY_NAME["gelu_tanh"]
    Y, A = torch.empty(M, h, dtype=torch.bfloat16, device="cuda"), torch.empty(t, M, F // t, dtype=torch.bfloat16,
                                                                               device="cuda")
    fwd = lambda: L.tp_mlp_forward(inp["X"], M, h, F, t, act, w.Wup_p, w.b_up, w.Wdown_p, w.b_down, None, Y, None, A,
                                   0, None, 0)
    fwd()
    torch.cuda.synchronize()
    Y_eager, A_eager = Y.clone(), A.clone()
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            fwd()
    torch.cuda.current_stream().wait_stream(cs)
    for _ in range(3):
        Y.zero_()
        A.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(Y.view(torch.int16), Y_eager.view(torch.int16))
        assert torch.equal(A.view(torch.int16), A_eager.view(torch.int16))
    assert L.tp_get_device_status(check=False) == L.TP_OK


def _deinterleave(Z, group=128):
    """[t][M][2 Ft] with gate / up in alternating groups -> (gate, up), each [t][M][Ft]."""
    t, M, W = Z.shape
    z = Z.reshape(t, M, W // (2 * group), 2, group)
    return z[:, :, :, 0, :].reshape(t, M, W // 2), z[:, :, :, 1, :].reshape(t, M, W // 2)


@pytest.mark.parametrize("M,h,F,t", [(256, 512, 2048, 4), (200, 264, 1024, 2), (1, 128, 512, 4),
                                     (384, 1024, 4096, 8)])
def test_swiglu_mlp_parity(M, h, F, t):
    """Token-parallel SwiGLU MLP forward and backward ("(times 2 for SwiGLU)"): gate
    and up split by the same columns, the row-parallel half and the f / g sums as for
    GeLU; checked against the fp64 oracle, gradients in the packed layouts."""
    _check_swiglu_mlp(M, h, F, t)


@pytest.mark.parametrize("pair", ["0", "1"])
def test_swiglu_fused_epilogues_both_kernels(pair, monkeypatch):
    """silu(gate) * up and its gradient run in the GEMM epilogues of both the single-CTA and
    the CTA-pair kernel.  F / t = 384: the dgrad's last 256-column tile of dA is half past
    N, so its second gate / up group is skipped; M = 300 leaves a ragged row tile."""
    monkeypatch.setenv("TP_GEMM_PAIR", pair)
    _check_swiglu_mlp(300, 256, 768, 2)


def _check_swiglu_mlp(M, h, F, t):
    inp = I.swiglu_inputs(M, h, F, seed=11, dy=True)
    dev = {k: v.cuda() for k, v in inp.items()}
    ref = {k: f64(v) for k, v in inp.items()}
    w = T.SwiGLUWeights(dev["W_gate"], dev["W_up"], dev["W_down"], None, t)
    Y, Z, A = T.mlp_forward(dev["X"], w, "swiglu")
    g = T.mlp_backward(dev["dY"], dev["X"], Z, A, w, "swiglu")
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    o = O.swiglu_forward_sharded(ref["X"], ref["W_gate"], ref["W_up"], ref["W_down"], t)
    b = O.swiglu_backward_sharded(ref["dY"], ref["X"], ref["W_gate"], ref["W_up"], ref["W_down"], o, t)
    assert_close("Y", f64(Y), o["Y"])
    assert_close("A", f64(A), np.stack(o["A"]))
    zg, zu = _deinterleave(f64(Z))
    assert_close("Z gate", zg, np.stack(o["Zg"]))
    assert_close("Z up", zu, np.stack(o["Zu"]))
    assert_close("dX", f64(g["dX"]), b["dX"])
    dWgu = O.pack_swiglu_weight(b["dW_gate"], b["dW_up"], t).reshape(t, 2 * F // t, h)
    assert_close("dW_gate/up (packed)", f64(g["dWup_p"]), dWgu)
    assert_close("dW_down (packed)", f64(g["dWdown_p"]), O.pack_row_weight(b["dW_down"], t))
    assert_close("db_down", f64(g["dbdown"]), ref["dY"].sum(axis=0))


def test_swiglu_mlp_argument_errors():
    M, h, F, t = 64, 128, 1024, 4
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    act = L.ACT_BY_NAME["swiglu"]
    # a gate / up bias is not part of this SwiGLU; F/t must be a multiple of the 128-row groups
    assert L.tp_mlp_forward(x, M, h, F, t, act, x, x, x, None, None, x, x, x, 0, None, 0,
                            check=False) == L.TP_ERR_UNSUPPORTED
    assert L.tp_mlp_forward(x, M, h, 4 * 192, t, act, x, None, x, None, None, x, x, x, 0, None, 0,
                            check=False) == L.TP_ERR_SHAPE
    # Z_save is required (the backward reads the gate and up pre-activations)
    assert L.tp_mlp_forward(x, M, h, F, t, act, x, None, x, None, None, x, None, x, 0, None, 0,
                            check=False) == L.TP_ERR_INVALID_ARG


def test_swiglu_autograd_function_accumulates():
    """TPMLPFunction with act="swiglu": dX equals the direct backward, and a second
    backward adds to the packed weight gradients kept on the weights object."""
    M, h, F, t = 128, 256, 1024, 4
    inp = I.swiglu_inputs(M, h, F, seed=17, dy=True)
    dev = {k: v.cuda() for k, v in inp.items()}
    w = T.SwiGLUWeights(dev["W_gate"], dev["W_up"], dev["W_down"], None, t)
    _, Z, A = T.mlp_forward(dev["X"], w, "swiglu")
    ref = T.mlp_backward(dev["dY"], dev["X"], Z, A, w, "swiglu")
    X = dev["X"].clone().requires_grad_(True)
    for _ in range(2):
        Y = T.TPMLPFunction.apply(X, w, "swiglu")
        (dx,) = torch.autograd.grad(Y, X, dev["dY"])
        assert torch.equal(dx.view(torch.int16), ref["dX"].view(torch.int16))
    torch.cuda.synchronize()
    assert w.grads["dbup"] is None
    for k in ("dWup_p", "dWdown_p", "dbdown"):
        assert torch.allclose(w.grads[k], 2 * ref[k], rtol=1e-5, atol=1e-6), k
