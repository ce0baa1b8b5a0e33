"""The C-ABI library loads, exports every symbol include/*.h declares, the
Python binding covers exactly those, and host-side argument validation
returns the documented status codes before any device work (no GPU needed)."""

import glob
import os
import re

import pytest

from megatron_tensor_transformer_shard_gb300 import _lib as L
from megatron_tensor_transformer_shard_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built_lib():
    B.build()
    return L.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^[A-Za-z_][\w \*]*?\b(tp_\w+)\s*\(", src, flags=re.M))
    return names


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) >= 15
    lib = L.lib()
    missing = [n for n in sorted(names) if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_header():
    assert declared_functions() == set(L.SIGNATURES)


def test_version_and_strings():
    assert L.tp_abi_version() == 1
    for code in range(8):
        assert L.status_string(code).startswith(("TP_OK", "TP_ERR"))


def test_workspace_sizes():
    # forward: the flags' partials, then room for the GEMMs' split-K partials (256 KB per
    # slot of up to 256, plus 64 bytes of counters each)
    sk = 256 * (256 * 256 * 4 + 64)
    assert L.tp_mlp_workspace_size(2048, 4096, 16384, 4, 0) == sk
    assert L.tp_mlp_workspace_size(2048, 4096, 16384, 4, L.TP_FLAG_UNFUSED_REDUCE) == 4 * 2048 * 4096 * 4 + sk
    assert L.tp_row_parallel_workspace_size(2048, 16384, 4096, 4) == sk
    assert L.tp_column_parallel_workspace_size(2048, 4096, 16384, 4) == sk
    assert L.tp_attn_forward_workspace_size(2048, 12288, 96, 128, 8, 0) == sk
    assert L.tp_mlp_backward_workspace_size(2048, 4096, 16384, 4, 0) >= 2048 * 16384 * 2
    # dZ (room for SwiGLU's gate and up) + db_down's partials + db_up's per-32-row partials that
    # the dgrad epilogue writes ([t][ceil(M / 32)][F / t] fp32), for ragged M as well
    for M, h, F, t in [(2048, 4096, 16384, 4), (200, 264, 784, 2), (1, 64, 128, 4), (33, 128, 1024, 8)]:
        need = M * F * 2 * 2 + t * ((M + 31) // 32) * (F // t) * 4 + ((M + 255) // 256) * h * 4
        assert L.tp_mlp_backward_workspace_size(M, h, F, t, 0) >= need, (M, h, F, t)
    assert L.tp_colsum_workspace_size(2048, 4096) == 32 * 4096 * 4
    # overlapped reduction: the t partials [t][M][h] fp32, then per 256 x 256 output tile an
    # fp32 running sum and 8 flags of 8 bytes
    assert L.tp_row_parallel_overlap_workspace_size(2048, 16384, 4096, 4) == \
        4 * 2048 * 4096 * 4 + 128 * (256 * 256 * 4 + 64)
    assert L.tp_row_parallel_overlap_workspace_size(300, 1024, 264, 3) == \
        (3 * 300 * 264 * 4 + 255) // 256 * 256 + 4 * (256 * 256 * 4 + 64)


def test_host_validation_without_device():
    c = dict(check=False, stream=0)
    # null input with tokens to process
    assert L.tp_mlp_forward(None, 4, 64, 128, 2, 2, 16, None, 16, None, None, 16, None, 16, 0, None, 0, **c) \
        == L.TP_ERR_INVALID_ARG
    # t does not divide F
    assert L.tp_mlp_forward(16, 4, 64, 128, 3, 2, 16, None, 16, None, None, 16, None, 16, 0, None, 0, **c) \
        == L.TP_ERR_SHAPE
    # hidden size not a multiple of 8
    assert L.tp_mlp_forward(16, 4, 60, 128, 2, 2, 16, None, 16, None, None, 16, None, 16, 0, None, 0, **c) \
        == L.TP_ERR_ALIGN
    # unknown activation
    assert L.tp_mlp_forward(16, 4, 64, 128, 2, 9, 16, None, 16, None, None, 16, None, 16, 0, None, 0, **c) \
        == L.TP_ERR_INVALID_ARG
    # no tokens: nothing to do
    assert L.tp_mlp_forward(None, 0, 64, 128, 2, 2, None, None, None, None, None, None, None, None, 0, None, 0,
                            **c) == L.TP_OK
    # unfused reduction without workspace
    assert L.tp_mlp_forward(16, 4, 64, 128, 2, 2, 16, None, 16, None, None, 16, None, 16,
                            L.TP_FLAG_UNFUSED_REDUCE, None, 0, **c) == L.TP_ERR_WORKSPACE
    # packing: t does not divide F
    assert L.tp_pack_col(16, 64, 100, 3, 16, **c) == L.TP_ERR_SHAPE
    assert L.tp_pack_qkv_heads(16, 96, 4, 16, 2, 16, **c) == L.TP_ERR_SHAPE
    assert L.tp_selftest_bounded_wait(0, **c) == L.TP_ERR_INVALID_ARG


def test_decode_attn_host_validation():
    c = dict(check=False, stream=0)
    ok_ws = L.tp_decode_attn_workspace_size(2, 1024, 8, 2, 128, 4, 256)
    assert ok_ws > 0
    assert L.tp_decode_attn_workspace_size(2, 1024, 8, 2, 64, 4, 256) == 0     # head_dim != 128
    assert L.tp_decode_attn_workspace_size(2, 1024, 8, 3, 128, 4, 256) == 0    # 3 KV heads do not group 8 heads
    args = lambda B, nh, nkv, hd, t, ws, nws: (16, B, nh * 128, nh, nkv, hd, t, 0.1, 16, None, 16, None, 16, 16,
                                               256, 16, 16, ws, nws)
    assert L.tp_decode_attn_forward(*args(2, 8, 2, 64, 4, 256, ok_ws), **c) == L.TP_ERR_SHAPE
    assert L.tp_decode_attn_forward(*args(2, 8, 2, 128, 3, 256, ok_ws), **c) == L.TP_ERR_SHAPE   # t does not divide
    assert L.tp_decode_attn_forward(*args(2, 12, 3, 128, 2, 256, ok_ws), **c) == L.TP_ERR_SHAPE  # 3 KV over 2 shards
    assert L.tp_decode_attn_forward(*args(0, 8, 2, 128, 4, None, 0), **c) == L.TP_OK             # nothing to do
    assert L.tp_decode_attn_forward(*args(2, 8, 2, 128, 4, 256 + 16, ok_ws), **c) == L.TP_ERR_ALIGN
    assert L.tp_decode_attn_forward(*args(2, 8, 2, 128, 4, 256, ok_ws - 256), **c) == L.TP_ERR_WORKSPACE
    assert L.tp_pack_qkv_gqa(16, 256, 8, 3, 128, 4, 16, **c) == L.TP_ERR_SHAPE
