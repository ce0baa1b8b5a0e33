"""GPU parity of decode attention over a head-sharded KV cache (grouped-query
heads sharded by KV group, replicated KV heads when n_kv < t) against the fp64
oracle, through the C ABI: max|gpu - oracle| <= 1e-2 max|oracle| for y and the
appended cache entries, bit-exact for every cache byte the call must not touch."""

import numpy as np
import pytest
import torch

import oracle as O
from megatron_tensor_transformer_shard_gb300 import _lib as L
from megatron_tensor_transformer_shard_gb300 import inputs as I
from megatron_tensor_transformer_shard_gb300 import tp as T

from gpu_helpers import assert_close, f64

pytestmark = pytest.mark.gpu

HD = 128


def _kv_first(nh, nkv, t, i):
    """First KV head held by shard i (the header's layout rule)."""
    return i * (nkv // t) if nkv >= t else (i * nkv) // t


def _shard_cache(C, nh, nkv, t):
    """Unsplit cache [n_kv][B][L][HD] -> per-shard copies [t][kv_t][B][L][HD] (device)."""
    kv_t = nkv // t if nkv >= t else 1
    idx = [_kv_first(nh, nkv, t, i) + j for i in range(t) for j in range(kv_t)]
    S = C.index_select(0, torch.tensor(idx)).contiguous()
    return S.view(t, kv_t, *C.shape[1:]).cuda()


def _f16_f64(t):
    return t.detach().cpu().double().numpy()


def _case(B, nh, nkv, t, L_max, pos, bias=True, seed=0, poison=False):
    d = nh * HD
    inp = I.decode_attn_inputs(B, d, nh, nkv, HD, L_max, bias=bias, seed=seed)
    w = T.DecodeAttnWeights(inp["W_qkv"].cuda(), None if inp["b_qkv"] is None else inp["b_qkv"].cuda(),
                            inp["W_o"].cuda(), None if inp["b_o"] is None else inp["b_o"].cuda(), nh, nkv, HD, t)
    Kd, Vd = _shard_cache(inp["K"], nh, nkv, t), _shard_cache(inp["V"], nh, nkv, t)
    posd = torch.tensor(pos, dtype=torch.int32).cuda()
    if poison:
        # bytes past the sequence end may hold anything: make them NaN / Inf
        for b, p in enumerate(pos):
            Kd[:, :, b, p:].view(torch.int16).fill_(0x7E00)
            Vd[:, :, b, p:].view(torch.int16).fill_(0x7C00)
    K0, V0 = Kd.clone(), Vd.clone()
    y = T.decode_attn_forward(inp["x"].cuda(), w, Kd, Vd, posd)
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    ref = O.decode_attn_sharded(
        f64(inp["x"]), f64(inp["W_qkv"]), None if inp["b_qkv"] is None else f64(inp["b_qkv"]), f64(inp["W_o"]),
        None if inp["b_o"] is None else f64(inp["b_o"]),
        O.shard_kv_cache(_f16_f64(inp["K"]), nh, nkv, t), O.shard_kv_cache(_f16_f64(inp["V"]), nh, nkv, t),
        pos, nh, nkv, HD, HD ** -0.5, t)
    return y, Kd, Vd, K0, V0, ref


def _check_cache(Kd, K0, ref_K, pos):
    got = Kd.cpu()
    before = K0.cpu()
    for b, p in enumerate(pos):
        new = _f16_f64(got[:, :, b, p])
        assert_close(f"cache[.., {b}, {p}]", new, ref_K[:, :, b, p])
        # every other position is untouched, bit for bit
        for sl in (slice(0, p), slice(p + 1, None)):
            assert torch.equal(got[:, :, b, sl].view(torch.int16), before[:, :, b, sl].view(torch.int16))


@pytest.mark.parametrize("nh,nkv,t", [
    (8, 2, 2),   # GQA, 2 KV heads per... one per shard, group 4
    (8, 2, 4),   # GQA, replicated: each KV head on 2 shards
    (8, 2, 8),   # one query head per shard, KV heads replicated 4x
    (8, 8, 4),   # multi-head (n_kv = n_heads)
    (8, 1, 4),   # MQA
    (8, 4, 1),   # unsharded reference point
])
def test_decode_attn_parity(nh, nkv, t):
    pos = [0, 300, 699]   # 1, 3 and 6 tiles of 128 keys, ragged tails
    y, Kd, Vd, K0, V0, ref = _case(3, nh, nkv, t, 700, pos)
    assert_close("y", f64(y), ref["y"])
    _check_cache(Kd, K0, ref["K_shards"], pos)
    _check_cache(Vd, V0, ref["V_shards"], pos)


def test_decode_attn_group_of_32_heads():
    # MQA with 32 query heads on one shard: the 32-wide head group
    pos = [129, 5]
    y, Kd, Vd, K0, V0, ref = _case(2, 32, 1, 1, 260, pos, seed=3)
    assert_close("y", f64(y), ref["y"])
    _check_cache(Kd, K0, ref["K_shards"], pos)


def test_decode_attn_ignores_nonfinite_bytes_past_the_end():
    pos = [1, 130, 255]
    y, _, _, _, _, ref = _case(3, 8, 2, 4, 384, pos, seed=5, poison=True)
    assert np.isfinite(f64(y)).all()
    assert_close("y", f64(y), ref["y"])


def test_decode_attn_no_bias_many_sequences():
    # 11 sequences: the GEMVs run as a group of 8 then a group of 3
    pos = [int(p) for p in I.decode_positions(11, 0, 520, seed=2)]
    y, Kd, _, K0, _, ref = _case(11, 8, 2, 2, 521, pos, bias=False, seed=9)
    assert_close("y", f64(y), ref["y"])
    _check_cache(Kd, K0, ref["K_shards"], pos)


@pytest.mark.parametrize("nh,nkv,t", [(8, 8, 2), (8, 2, 4)])
def test_decode_steps_match_causal_prefill(nh, nkv, t):
    """Tokens fed one by one through the GPU cache reproduce the rows of causal
    prefill attention over the whole sequence (oracle)."""
    d, N, L_max = nh * HD, 140, 160
    inp = I.decode_attn_inputs(1, d, nh, nkv, HD, L_max, seed=11)
    X = I.attn_inputs(N, d, bias=False, dy=False, seed=12)["X"]
    w = T.DecodeAttnWeights(inp["W_qkv"].cuda(), inp["b_qkv"].cuda(), inp["W_o"].cuda(), inp["b_o"].cuda(),
                            nh, nkv, HD, t)
    kv_t = nkv // t if nkv >= t else 1
    Kd = torch.zeros(t, kv_t, 1, L_max, HD, dtype=torch.float16, device="cuda")
    Vd = torch.zeros_like(Kd)
    ws = w.workspace(1, L_max, "cuda")
    Xd = X.cuda()
    ys = []
    for n in range(N):
        ys.append(T.decode_attn_forward(Xd[n:n + 1], w, Kd, Vd, torch.tensor([n], dtype=torch.int32).cuda(), ws=ws))
    torch.cuda.synchronize()
    assert L.tp_get_device_status(check=False) == L.TP_OK
    full = O.attn_gqa_forward_unsplit(f64(X), f64(inp["W_qkv"]), f64(inp["b_qkv"]), f64(inp["W_o"]),
                                      f64(inp["b_o"]), nh, nkv, HD, True, HD ** -0.5)["Y"]
    assert_close("decode rows", np.concatenate([f64(y) for y in ys]), full)


def test_decode_attn_graph_replay_matches_eager():
    """The step launches through programmatic dependent launches; captured in a
    CUDA graph and replayed it gives the same bits as the eager call."""
    nh, nkv, t, B, L_max = 8, 2, 2, 4, 640
    d = nh * HD
    inp = I.decode_attn_inputs(B, d, nh, nkv, HD, L_max, seed=21)
    w = T.DecodeAttnWeights(inp["W_qkv"].cuda(), inp["b_qkv"].cuda(), inp["W_o"].cuda(), inp["b_o"].cuda(),
                            nh, nkv, HD, t)
    Kd, Vd = _shard_cache(inp["K"], nh, nkv, t), _shard_cache(inp["V"], nh, nkv, t)
    posd = torch.tensor([5, 200, 639, 333], dtype=torch.int32).cuda()
    x = inp["x"].cuda()
    ws = w.workspace(B, L_max, "cuda")
    y_eager = T.decode_attn_forward(x, w, Kd, Vd, posd, ws=ws).clone()
    y = torch.empty_like(y_eager)
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cs):
        with torch.cuda.graph(g, stream=cs):
            T.decode_attn_forward(x, w, Kd, Vd, posd, ws=ws, out=y)
    torch.cuda.current_stream().wait_stream(cs)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y_eager.view(torch.int16))
    assert L.tp_get_device_status(check=False) == L.TP_OK


def test_decode_attn_position_out_of_range_is_reported():
    nh, nkv, t, B, L_max = 8, 2, 2, 2, 256
    d = nh * HD
    inp = I.decode_attn_inputs(B, d, nh, nkv, HD, L_max, seed=4)
    w = T.DecodeAttnWeights(inp["W_qkv"].cuda(), None, inp["W_o"].cuda(), None, nh, nkv, HD, t)
    Kd, Vd = _shard_cache(inp["K"], nh, nkv, t), _shard_cache(inp["V"], nh, nkv, t)
    K0 = Kd.clone()
    T.decode_attn_forward(inp["x"].cuda(), w, Kd, Vd, torch.tensor([3, L_max], dtype=torch.int32).cuda())
    assert L.tp_get_device_status(check=False) == L.TP_ERR_SHAPE
    # the out-of-range sequence's cache is untouched; the context stays usable
    assert torch.equal(Kd[:, :, 1].view(torch.int16), K0[:, :, 1].view(torch.int16))
    T.decode_attn_forward(inp["x"].cuda(), w, Kd, Vd, torch.tensor([3, 4], dtype=torch.int32).cuda())
    assert L.tp_get_device_status(check=False) == L.TP_OK


def test_decode_pack_matches_oracle_layout():
    for nh, nkv, t in [(8, 2, 4), (8, 2, 8), (8, 8, 2), (16, 4, 2)]:
        d = 256
        g = torch.Generator().manual_seed(nh * 100 + nkv * 10 + t)
        W = torch.randn(d, (nh + 2 * nkv) * HD, generator=g).to(torch.bfloat16)
        b = torch.randn((nh + 2 * nkv) * HD, generator=g).to(torch.bfloat16)
        w = T.DecodeAttnWeights(W.cuda(), b.cuda(), torch.zeros(nh * HD, d, dtype=torch.bfloat16).cuda(), None,
                                nh, nkv, HD, t)
        want = O.pack_qkv_gqa_weight(I.bits(W), nh, nkv, HD, t)
        assert np.array_equal(I.bits(w.Wqkv_p.cpu()), want)
        assert np.array_equal(I.bits(w.bqkv_p.cpu()), O.pack_qkv_gqa_bias(I.bits(b), nh, nkv, HD, t))
        back = torch.empty_like(W).cuda()
        L.tp_unpack_qkv_gqa(w.Wqkv_p, d, nh, nkv, HD, t, back)
        torch.cuda.synchronize()
        assert torch.equal(back.cpu().view(torch.int16), W.view(torch.int16))


@pytest.mark.slow
def test_decode_attn_full_size():
    """Llama-3-70B-shaped attention at TP=4 (64 query heads, 8 KV heads), 8
    sequences with cache lengths between 4096 and 8192 keys."""
    nh, nkv, t, B, L_max = 64, 8, 4, 8, 8192
    pos = [int(p) for p in I.decode_positions(B, 4095, L_max - 1, seed=0)]
    y, Kd, _, K0, _, ref = _case(B, nh, nkv, t, L_max, pos, bias=False, seed=0)
    assert_close("y", f64(y), ref["y"])
    got = Kd.cpu()
    for b, p in enumerate(pos):
        assert_close(f"cache {b}", _f16_f64(got[:, :, b, p]), ref["K_shards"][:, :, b, p])
