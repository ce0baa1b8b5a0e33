"""GPU parity of the vocab-parallel embedding through the C ABI: the lookup
is bit-exact (it moves bf16 bits), the gradient matches the fp64 oracle within
max|gpu - oracle| <= 1e-2 max|oracle| and is deterministic run to run."""

import numpy as np
import pytest
import torch

import oracle as O
from megatron_tensor_transformer_shard_gb300 import _lib as L
from megatron_tensor_transformer_shard_gb300 import inputs as I

from gpu_helpers import assert_close, f64

pytestmark = pytest.mark.gpu


def _fwd(ids, E, V, h, t):
    Y = torch.empty(ids.numel(), h, dtype=torch.bfloat16, device="cuda")
    L.tp_vocab_embedding_forward(ids, ids.numel(), V, h, t, E, Y)
    return Y


def _bwd(ids, dY, V, h, t, dE=None, accumulate=0):
    N = ids.numel()
    if dE is None:
        dE = torch.empty(V, h, dtype=torch.float32, device="cuda")
    nws = L.tp_vocab_embedding_backward_workspace_size(N)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")
    L.tp_vocab_embedding_backward(ids, dY, N, V, h, t, dE, accumulate, ws, ws.numel())
    return dE


@pytest.mark.parametrize("N,V,h,t", [(300, 64, 256, 4), (9000, 1000, 264, 8), (1, 16, 8, 2), (5000, 4096, 512, 1),
                                     (1500, 512, 128, 2), (2048, 96, 64, 4),
                                     (4000, 40000, 1032, 4),    # mostly ids seen once; three column slices
                                     (700, 2, 64, 2)])          # two ids: two long segments
def test_embedding_parity(N, V, h, t):
    ids = I.token_ids(N, V, seed=N)
    ids[:4] = torch.tensor([0, V - 1, V // t - 1, min(V // t, V - 1)], dtype=torch.int32)[: min(4, N)]
    inp = I.embedding_inputs(N, V, h, seed=V)
    idd, E, dY = ids.cuda(), inp["E"].cuda(), inp["dY"].cuda()
    Y = _fwd(idd, E, V, h, t)
    dE = _bwd(idd, dY, V, h, t)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    # forward: exact bits of the owning shard's row
    assert torch.equal(Y.cpu().view(torch.int16), inp["E"][ids.long()].view(torch.int16))
    ref = O.embedding_forward_sharded(ids.numpy(), f64(inp["E"]), t)["Y"]
    assert np.array_equal(f64(Y), ref)
    # backward: per-shard gradients, untouched rows exactly zero
    parts = O.embedding_backward_sharded(ids.numpy(), f64(inp["dY"]), V, t) if N <= 5000 else None
    want = np.concatenate(parts) if parts is not None else O.embedding_backward_unsplit(ids.numpy(), f64(inp["dY"]), V)
    got = f64(dE)
    assert_close("dE", got, want)
    untouched = np.setdiff1d(np.arange(V), ids.numpy())
    assert (got[untouched] == 0).all()


def test_embedding_backward_deterministic_and_accumulates():
    N, V, h, t = 12000, 500, 128, 4   # two sorted chunks, many repeats
    ids = I.token_ids(N, V, zipf_s=1.3, seed=7)
    inp = I.embedding_inputs(N, V, h, seed=8)
    idd, dY = ids.cuda(), inp["dY"].cuda()
    a = _bwd(idd, dY, V, h, t).clone()
    b = _bwd(idd, dY, V, h, t).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    c = _bwd(idd, dY, V, h, t, dE=b, accumulate=1)   # b + grad
    torch.cuda.synchronize()
    assert_close("accumulated", f64(c), 2 * O.embedding_backward_unsplit(ids.numpy(), f64(inp["dY"]), V))


def test_embedding_id_out_of_range_is_reported():
    V, h, t = 32, 16, 2
    E = torch.randn(V, h).to(torch.bfloat16).cuda()
    ids = torch.tensor([3, V, 5], dtype=torch.int32).cuda()
    Y = _fwd(ids, E, V, h, t)
    assert L.tp_get_device_status(check=False) == L.TP_ERR_SHAPE
    assert (Y[1].float() == 0).all() and torch.equal(Y[0], E[3])
    dY = torch.ones(3, h, dtype=torch.bfloat16, device="cuda")
    dE = _bwd(ids, dY, V, h, t)
    assert L.tp_get_device_status(check=False) == L.TP_ERR_SHAPE
    assert dE[3].eq(1).all() and dE[5].eq(1).all() and dE.sum().item() == 2 * h


def test_embedding_backward_skips_out_of_range_ids_among_many():
    """Ids outside [0, V) spread through a chunk (negative and too large) are reported
    and add nothing; every other token's row is summed as the oracle sums the valid
    tokens alone."""
    N, V, h, t = 3000, 700, 520, 4
    ids = I.token_ids(N, V, seed=11)
    bad = torch.arange(5, N, 97)
    ids[bad] = torch.where(bad % 2 == 0, torch.full_like(bad, -3), torch.full_like(bad, V + 5)).to(torch.int32)
    inp = I.embedding_inputs(N, V, h, seed=12)
    dE = _bwd(ids.cuda(), inp["dY"].cuda(), V, h, t)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_ERR_SHAPE
    ok = ((ids >= 0) & (ids < V)).numpy()
    want = O.embedding_backward_unsplit(ids.numpy()[ok], f64(inp["dY"])[ok], V)
    assert_close("dE", f64(dE), want)


def test_embedding_rejects_bad_shapes():
    x = torch.zeros(16, dtype=torch.int32, device="cuda")
    y = torch.zeros(16, 8, dtype=torch.bfloat16, device="cuda")
    assert L.tp_vocab_embedding_forward(x, 16, 30, 8, 4, y, y, check=False) == L.TP_ERR_SHAPE     # t does not divide V
    assert L.tp_vocab_embedding_forward(x, 16, 1 << 19, 8, 1, y, y, check=False) == L.TP_ERR_SHAPE
    assert L.tp_vocab_embedding_forward(x, 16, 32, 12, 4, y, y, check=False) == L.TP_ERR_ALIGN


@pytest.mark.slow
def test_embedding_full_size():
    """Llama-3-sized vocabulary (128256) x 8192 at TP=4, 4096 Zipf-distributed tokens."""
    N, V, h, t = 4096, 128256, 8192, 4
    ids = I.token_ids(N, V, seed=0)
    inp = I.embedding_inputs(N, V, h, seed=0, device="cuda")
    idd = ids.cuda()
    Y = _fwd(idd, inp["E"], V, h, t)
    dE = _bwd(idd, inp["dY"], V, h, t)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    assert torch.equal(Y.view(torch.int16), inp["E"][idd.long()].view(torch.int16))
    uniq = torch.unique(idd.long())
    want = O.embedding_backward_unsplit(ids.numpy(), f64(inp["dY"]), V)[uniq.cpu().numpy()]
    assert_close("dE touched rows", dE[uniq].double().cpu().numpy(), want)
    sample = torch.randint(0, V, (2000,), generator=torch.Generator().manual_seed(1)).cuda()
    sample = sample[~torch.isin(sample, uniq)]
    assert (dE[sample] == 0).all()
