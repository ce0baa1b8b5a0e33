"""The pages' own small checks, rebuilt: the oracle's sharded forward and
backward are compared with torch autograd in float64 on the same toy set-ups
the pages use (seed, shapes, scaling, loss).  Autograd is independent of the
oracle's hand-written backward, which is what makes these pins.

* "Parallelism Strategies #1 - Tensor Parallelism": 3x3 FFN with no
  activation, ``torch.manual_seed(42)``, ``torch.rand`` inputs, weights in
  PyTorch (out, in) form, loss mean(Y); the shard grads vstack/hstack to the
  full weight grads.
* "Tensor and sequence parallelism" (section "The implementation",
  tp_mlp_check.py): TP=4, S=8, H=16, FFN=64, seed 0, ``randn`` with
  w1/sqrt(H), w2/sqrt(FFN), LayerNorm with weight only, GeLU (erf), loss
  sum(out^2); TP and TP+SP variants, including the all-reduce of the
  LayerNorm weight grad.
"""

import numpy as np
import torch
import torch.nn.functional as F

import oracle as O


def test_first_page_toy_structure():
    torch.manual_seed(42)
    X = torch.rand(3, 3, dtype=torch.float32).double()
    W1 = torch.rand(2, 3, dtype=torch.float32).double()   # (out, in)
    W2 = torch.rand(3, 2, dtype=torch.float32).double()
    Xr, W1r, W2r = (v.clone().requires_grad_() for v in (X, W1, W2))
    Y = (Xr @ W1r.t()) @ W2r.t()
    Y.mean().backward()
    # oracle in X @ W form: W_up = W1^T, W_down = W2^T, identity activation, t = 2
    x, wu, wd = X.numpy(), W1.numpy().T.copy(), W2.numpy().T.copy()
    f = O.mlp_forward_sharded(x, wu, None, wd, None, "identity", 2)
    assert np.allclose(f["Y"], Y.detach().numpy(), rtol=0, atol=1e-14)
    assert np.allclose(np.concatenate(f["A"], axis=1), (Xr @ W1r.t()).detach().numpy(), atol=1e-15)
    G = np.ones((3, 3)) / 9.0                       # d mean(Y) / dY
    b = O.mlp_backward_sharded(G, x, wu, wd, f, "identity", 2)
    assert np.allclose(b["dX"], Xr.grad.numpy(), atol=1e-15)
    assert np.allclose(sum(b["dX_partials"]), Xr.grad.numpy(), atol=1e-15)
    # shard grads of W1 (rows in (out, in) form) stack vertically, those of W2 horizontally
    dW1_shards = [b["dW_up"][:, O.shard_slice(2, 2, i)].T for i in range(2)]
    dW2_shards = [b["dW_down"][O.shard_slice(2, 2, i), :].T for i in range(2)]
    assert np.allclose(np.vstack(dW1_shards), W1r.grad.numpy(), atol=1e-15)
    assert np.allclose(np.hstack(dW2_shards), W2r.grad.numpy(), atol=1e-15)


def _p4_setup():
    S, H, FFN, tp = 8, 16, 64, 4
    torch.manual_seed(0)
    x_full = torch.randn(S, H)
    ln_w = torch.randn(H)
    w1 = torch.randn(FFN, H) / H ** 0.5
    w2 = torch.randn(H, FFN) / FFN ** 0.5
    return S, H, FFN, tp, x_full.double(), ln_w.double(), w1.double(), w2.double()


def test_handbook_tp_check():
    S, H, FFN, tp, x_full, ln_w, w1, w2 = _p4_setup()
    ins = [v.clone().requires_grad_() for v in (x_full, ln_w, w1, w2)]
    h = F.layer_norm(ins[0], (H,), weight=ins[1])
    out = F.linear(F.gelu(F.linear(h, ins[2])), ins[3])
    out.square().sum().backward()
    r_x, r_ln, r_w1, r_w2 = (v.grad.numpy() for v in ins)

    x, g, W_up, W_down = x_full.numpy(), ln_w.numpy(), w1.numpy().T.copy(), w2.numpy().T.copy()
    zero = np.zeros(H)
    y_ln, m, r = O.layernorm_forward(x, g, zero, 1e-5)
    f = O.mlp_forward_sharded(y_ln, W_up, None, W_down, None, "gelu_erf", tp)
    assert np.abs(f["Y"] - out.detach().numpy()).max() < 1e-12
    G = 2.0 * f["Y"]                                 # d sum(out^2) / d out
    b = O.mlp_backward_sharded(G, y_ln, W_up, W_down, f, "gelu_erf", tp)
    dx, dg, _ = O.layernorm_backward(b["dX"], x, g, m, r)
    assert np.abs(dx - r_x).max() < 1e-12
    assert np.abs(dg - r_ln).max() < 1e-12
    for rank in range(tp):
        cols = O.shard_slice(FFN, tp, rank)
        assert np.abs(b["dW_up"][:, cols].T - r_w1[cols]).max() < 1e-12        # w1_s.grad
        assert np.abs(b["dW_down"][cols, :].T - r_w2[:, cols]).max() < 1e-12   # w2_s.grad


def test_handbook_sp_check():
    S, H, FFN, tp, x_full, ln_w, w1, w2 = _p4_setup()
    ins = [v.clone().requires_grad_() for v in (x_full, ln_w, w1, w2)]
    h = F.layer_norm(ins[0], (H,), weight=ins[1])
    ref_out = F.linear(F.gelu(F.linear(h, ins[2])), ins[3])
    ref_out.square().sum().backward()
    r_x, r_ln = ins[0].grad.numpy(), ins[1].grad.numpy()

    x, g = x_full.numpy(), ln_w.numpy()
    W_up, W_down = w1.numpy().T.copy(), w2.numpy().T.copy()
    zero = np.zeros(H)
    Xs = x.reshape(tp, S // tp, H)                   # rows = slice(rank*S//tp, ...)
    ys, ms, rs = O.sp_layernorm_forward(Xs, g, zero, 1e-5)
    hfull = O.all_gather_seq(ys)                     # GatherSeq forward
    f = O.mlp_forward_sharded(hfull, W_up, None, W_down, None, "gelu_erf", tp)
    out_sh = O.reduce_scatter_seq(f["P"], tp)        # ScatterSeq forward
    ref = ref_out.detach().numpy()
    for rank in range(tp):
        assert np.abs(out_sh[rank] - ref[O.shard_slice(S, tp, rank)]).max() < 1e-12
    Gsh = 2.0 * out_sh
    Gfull = O.all_gather_seq(Gsh)                    # ScatterSeq backward
    b = O.mlp_backward_sharded(Gfull, hfull, W_up, W_down, f, "gelu_erf", tp)
    dh_sh = O.reduce_scatter_seq(b["dX_partials"], tp)   # GatherSeq backward
    dxs, dgp, _, dg, _ = O.sp_layernorm_backward(dh_sh, Xs, g, ms, rs)
    for rank in range(tp):
        assert np.abs(dxs[rank] - r_x[O.shard_slice(S, tp, rank)]).max() < 1e-12
    # each rank's own LayerNorm weight grad is only a part; the sum is the full grad
    assert np.abs(dgp[0] - r_ln).max() > 1e-6
    assert np.abs(dg - r_ln).max() < 1e-12
