"""tp_colsum_noalloc -- column sums for callers that cannot allocate device
memory (no cudaMalloc allowed, or all device memory already owned by another
allocator), so they cannot pass the workspace tp_colsum needs.  Its scratch is
a fixed array inside the library.  Checked against tp_colsum, through the C
ABI, on two calls in a row (the second reuses the array the first one wrote).

This file is named to be collected last, and passes both alone in a fresh
process and after the other GPU tests."""

import numpy as np
import pytest
import torch

from megatron_tensor_transformer_shard_gb300 import _lib as L

from gpu_helpers import TOL, rel_err

pytestmark = pytest.mark.gpu


def _with_workspace(G, rows, cols):
    out = torch.empty(cols, dtype=torch.float32, device="cuda")
    nws = L.tp_colsum_workspace_size(rows, cols)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")
    L.tp_colsum(G, rows, cols, out, 0, ws, nws)
    return out


def _fp64_colsum(G):
    """The plain definition: every column's sum over all rows, in float64 on the host."""
    return G.cpu().double().numpy().sum(axis=0)


def test_noalloc_matches_workspace_version_twice():
    shapes = [(2048, 4096), (333, 1026)]       # second call: other sizes, ragged rows
    for k, (rows, cols) in enumerate(shapes):
        g = torch.Generator().manual_seed(40 + k)
        G = torch.randn(rows, cols, generator=g).to(torch.bfloat16).cuda()
        ref = _with_workspace(G, rows, cols)
        out = torch.full((cols,), float("nan"), dtype=torch.float32, device="cuda")
        L.tp_colsum_noalloc(G, rows, cols, out, 0)
        torch.cuda.synchronize()
        assert L.tp_get_device_status(check=False) == L.TP_OK
        a, b = out.double().cpu().numpy(), ref.double().cpu().numpy()
        assert np.all(np.isfinite(a))
        assert rel_err(a, b) <= TOL
        assert np.array_equal(a, b)               # same reduction order -> identical sums
        assert rel_err(a, _fp64_colsum(G)) <= TOL  # and both are the column sums


def test_noalloc_more_chunks_than_grid_y():
    """More 64-row chunks (70001) than a grid's y dimension holds (65535): the chunks
    are spread over x, and both entry points still give the column sums."""
    rows, cols = 64 * 70000 + 5, 2
    G = torch.randn(rows, cols, generator=torch.Generator().manual_seed(44)).to(torch.bfloat16).cuda()
    out = torch.full((cols,), float("nan"), dtype=torch.float32, device="cuda")
    L.tp_colsum_noalloc(G, rows, cols, out, 0)
    ref = _with_workspace(G, rows, cols)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    a, b = out.double().cpu().numpy(), ref.double().cpu().numpy()
    exact = _fp64_colsum(G)
    assert np.array_equal(a, b)
    # fp32 sums of 4.5M N(0,1) terms: the sum's spread is ~2100, the fp32 rounding far smaller
    assert np.abs(a - exact).max() <= 1e-3 * np.abs(G.cpu().double().numpy()).sum(axis=0).max()


def test_noalloc_accumulate_and_limit():
    rows, cols = 512, 2048
    G = torch.randn(rows, cols, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16).cuda()
    base = torch.randn(cols, generator=torch.Generator().manual_seed(8)).cuda()
    out = base.clone()
    L.tp_colsum_noalloc(G, rows, cols, out, 1)
    ref = base + _with_workspace(G, rows, cols)
    torch.cuda.synchronize()
    assert rel_err(out.double().cpu().numpy(), ref.double().cpu().numpy()) <= TOL
    # beyond the fixed scratch (ceil(rows/64) * cols > 2^20 floats) the call is refused
    assert L.tp_colsum_noalloc(G, 64 * 64 + 1, 16384, out, 0, check=False) == L.TP_ERR_SHAPE
