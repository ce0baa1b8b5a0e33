"""GPU parity of the decode SwiGLU GEMV and the sequence-parallel LayerNorm
against the fp64 oracle, through the C ABI (max|gpu - oracle| <= 1e-2 max|oracle|)."""

import numpy as np
import pytest
import torch

import oracle as O
from megatron_tensor_transformer_shard_gb300 import _lib as L
from megatron_tensor_transformer_shard_gb300 import inputs as I

from gpu_helpers import assert_close, f64

pytestmark = pytest.mark.gpu


def _decode(M, h, F, t, seed=0):
    inp = I.swiglu_inputs(M, h, F, seed=seed)
    dev = {k: v.cuda() for k, v in inp.items()}
    Wgu = torch.empty(2 * F, h, dtype=torch.bfloat16, device="cuda")
    Wd = torch.empty(t, h, F // t, dtype=torch.bfloat16, device="cuda")
    L.tp_pack_swiglu(dev["W_gate"], dev["W_up"], h, F, t, Wgu)
    L.tp_pack_row(dev["W_down"], F, h, t, Wd)
    y = torch.empty(M, h, dtype=torch.bfloat16, device="cuda")
    a = torch.empty(M, F, dtype=torch.bfloat16, device="cuda")
    L.tp_decode_swiglu_forward(dev["X"], M, h, F, t, Wgu, Wd, y, a)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    ref = {k: f64(v) for k, v in inp.items()}
    o = O.swiglu_forward_sharded(ref["X"], ref["W_gate"], ref["W_up"], ref["W_down"], t)
    assert_close("y", f64(y), o["Y"])
    assert_close("a", f64(a), np.concatenate(o["A"], axis=1))


@pytest.mark.parametrize("M,h,F,t", [(1, 256, 1024, 4), (3, 512, 2048, 2), (8, 264, 1024, 8), (1, 1024, 4096, 1)])
def test_decode_swiglu_parity(M, h, F, t):
    _decode(M, h, F, t)


@pytest.mark.slow
def test_decode_swiglu_full_size():
    c = I.CONFIGS["c3"]
    _decode(c["M"], c["h"], c["F"], c["t"])


def test_decode_rejects_bad_shapes():
    x = torch.zeros(1, 256, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(1, 256, dtype=torch.bfloat16, device="cuda")
    assert L.tp_decode_swiglu_forward(x, 9, 256, 1024, 4, x, x, y, y, check=False) == L.TP_ERR_SHAPE
    assert L.tp_decode_swiglu_forward(x, 1, 256, 1000, 4, x, x, y, y, check=False) == L.TP_ERR_SHAPE


def _ln(s, h, t, with_dres, seed=0):
    inp = I.ln_inputs(s, h, seed=seed)
    dev = {k: v.cuda() for k, v in inp.items()}
    Y = torch.empty(s, h, dtype=torch.bfloat16, device="cuda")
    mean = torch.empty(s, dtype=torch.float32, device="cuda")
    rstd = torch.empty(s, dtype=torch.float32, device="cuda")
    L.tp_sp_layernorm_forward(dev["X"], s, h, t, dev["gamma"], dev["beta"], 1e-5, Y, mean, rstd)
    dres = torch.randn(s, h, generator=torch.Generator().manual_seed(seed + 1)).to(torch.bfloat16)
    dX = torch.empty(s, h, dtype=torch.bfloat16, device="cuda")
    dgp = torch.empty(t, h, dtype=torch.float32, device="cuda")
    dbp = torch.empty(t, h, dtype=torch.float32, device="cuda")
    dg = torch.empty(h, dtype=torch.float32, device="cuda")
    db = torch.empty(h, dtype=torch.float32, device="cuda")
    L.tp_sp_layernorm_backward(dev["dY"], dev["X"], dev["gamma"], mean, rstd, dres.cuda() if with_dres else None,
                               s, h, t, dX, dgp, dbp, dg, db)
    torch.cuda.synchronize()
    ref = {k: f64(v) for k, v in inp.items()}
    Xs = ref["X"].reshape(t, s // t, h)
    ys, ms, rs = O.sp_layernorm_forward(Xs, ref["gamma"], ref["beta"], 1e-5)
    assert_close("Y", f64(Y), ys.reshape(s, h))
    assert_close("mean", f64(mean), ms.reshape(s))
    assert_close("rstd", f64(rstd), rs.reshape(s))
    dxs, dgp_r, dbp_r, dg_r, db_r = O.sp_layernorm_backward(ref["dY"].reshape(t, s // t, h), Xs, ref["gamma"],
                                                            ms, rs)
    dx_ref = dxs.reshape(s, h) + (f64(dres) if with_dres else 0.0)
    assert_close("dX", f64(dX), dx_ref)
    assert_close("dgamma_part", f64(dgp), dgp_r)
    assert_close("dbeta_part", f64(dbp), dbp_r)
    assert_close("dgamma", f64(dg), dg_r)
    assert_close("dbeta", f64(db), db_r)


@pytest.mark.parametrize("s,h,t,dres", [(64, 256, 4, False), (48, 1000 - 1000 % 8, 2, True), (8, 12288, 1, True),
                                        (512, 1024, 8, True)])
def test_sp_layernorm_parity(s, h, t, dres):
    _ln(s, h, t, dres)


# More shapes: shard row counts that are not multiples of the column kernel's 32-row
# step, a row of 4992 columns (a thread's last 8-column chunk past the end for some
# threads), 8192 columns with dres, and 16 shards.
@pytest.mark.parametrize("s,h,t,dres", [(320, 512, 8, False), (8 * 21, 4992, 8, True), (8 * 64, 8192, 8, True),
                                        (16 * 24, 768, 16, False)])
def test_sp_layernorm_more_shapes(s, h, t, dres):
    _ln(s, h, t, dres)


@pytest.mark.slow
def test_sp_layernorm_full_size():
    _ln(4096, 8192, 8, True)
