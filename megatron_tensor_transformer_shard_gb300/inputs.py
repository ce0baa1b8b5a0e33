"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no arithmetic of the method: it only draws float32 normals
from a seeded ``torch.Generator`` in a fixed tensor order, scales them by the
stated standard deviation and rounds them to bf16 (round-to-nearest-even).
Both the CUDA path and the oracle consume the resulting bits.

Workload shapes (the five configurations this library is measured on):

* ``c1``: TP MLP forward, t=2, X 128x1024, W_up 1024x4096, W_down 4096x1024.
* ``c2``: TP MLP forward+backward, t=4, X 2048x4096, W_up 4096x16384,
  W_down 16384x4096, dY 2048x4096.
* ``c3``: decode SwiGLU MLP, t=4, x 1x8192, W_gate/W_up 8192x28672,
  W_down 28672x8192, no biases.
* ``c4``: full TP layer, t=8, N=2048, d=12288, 96 heads x 128, MLP 4d, causal.
* ``c5``: sequence-parallel TP layer, t=8, s=4096, h=8192, 64 heads x 128,
  MLP 4h, causal.

Distributions: activations and dY ~ N(0,1); weights ~ N(0, 0.02) (standard
deviation 0.02); biases 0.01*N(0,1); LayerNorm gamma = 1 + N(0,0.02) and
beta = N(0,0.02).
"""

from __future__ import annotations

import numpy as np
import torch

WEIGHT_STD = 0.02
BIAS_SCALE = 0.01

CONFIGS = {
    "c1": dict(kind="mlp", M=128, h=1024, F=4096, t=2, act="gelu_tanh", bias=True, backward=False),
    "c2": dict(kind="mlp", M=2048, h=4096, F=16384, t=4, act="gelu_tanh", bias=True, backward=True),
    "c3": dict(kind="swiglu_decode", M=1, h=8192, F=28672, t=4, bias=False, backward=False),
    "c4": dict(kind="layer", N=2048, d=12288, n_heads=96, head_dim=128, F=49152, t=8, sp=False,
               act="gelu_tanh", causal=True, eps=1e-5, backward=True),
    "c5": dict(kind="layer", N=4096, d=8192, n_heads=64, head_dim=128, F=32768, t=8, sp=True,
               act="gelu_tanh", causal=True, eps=1e-5, backward=True),
}


def _draw(gen: torch.Generator, shape, scale: float, device) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32, device=device)
    if scale != 1.0:
        x = x * scale
    return x.to(torch.bfloat16)


def make_generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def mlp_inputs(M, h, F, bias=True, dy=True, seed=0, device="cpu"):
    """X, W_up (h, F), b_up, W_down (F, h), b_down, dY, drawn in that order."""
    g = make_generator(seed, device)
    out = {"X": _draw(g, (M, h), 1.0, device), "W_up": _draw(g, (h, F), WEIGHT_STD, device)}
    out["b_up"] = _draw(g, (F,), BIAS_SCALE, device) if bias else None
    out["W_down"] = _draw(g, (F, h), WEIGHT_STD, device)
    out["b_down"] = _draw(g, (h,), BIAS_SCALE, device) if bias else None
    out["dY"] = _draw(g, (M, h), 1.0, device) if dy else None
    return out


def swiglu_inputs(M, h, F, seed=0, device="cpu", dy=False):
    """x, W_gate (h, F), W_up (h, F), W_down (F, h), and dY (M, h) if asked, drawn in that order."""
    g = make_generator(seed, device)
    out = {"X": _draw(g, (M, h), 1.0, device), "W_gate": _draw(g, (h, F), WEIGHT_STD, device),
           "W_up": _draw(g, (h, F), WEIGHT_STD, device), "W_down": _draw(g, (F, h), WEIGHT_STD, device)}
    if dy:
        out["dY"] = _draw(g, (M, h), 1.0, device)
    return out


def attn_inputs(N, d, bias=True, dy=True, seed=0, device="cpu"):
    """Xn (N, d), W_qkv (d, 3d) laid out [Q|K|V], b_qkv, W_o (d, d), b_o, dY."""
    g = make_generator(seed, device)
    out = {"X": _draw(g, (N, d), 1.0, device), "W_qkv": _draw(g, (d, 3 * d), WEIGHT_STD, device)}
    out["b_qkv"] = _draw(g, (3 * d,), BIAS_SCALE, device) if bias else None
    out["W_o"] = _draw(g, (d, d), WEIGHT_STD, device)
    out["b_o"] = _draw(g, (d,), BIAS_SCALE, device) if bias else None
    out["dY"] = _draw(g, (N, d), 1.0, device) if dy else None
    return out


def ln_inputs(s, h, seed=0, device="cpu"):
    """X (s, h), gamma, beta, dY."""
    g = make_generator(seed, device)
    X = _draw(g, (s, h), 1.0, device)
    gamma = (1.0 + WEIGHT_STD * torch.randn(h, generator=g, device=device)).to(torch.bfloat16)
    beta = _draw(g, (h,), WEIGHT_STD, device)
    dY = _draw(g, (s, h), 1.0, device)
    return {"X": X, "gamma": gamma, "beta": beta, "dY": dY}


def layer_inputs(N, d, F, seed=0, device="cpu"):
    """Full layer: X, W_qkv, b_qkv, W_o, b_o, W_up, b_up, W_down, b_down,
    ln1 gamma/beta, ln2 gamma/beta, dY -- in that order."""
    g = make_generator(seed, device)
    out = {"X": _draw(g, (N, d), 1.0, device)}
    out["W_qkv"] = _draw(g, (d, 3 * d), WEIGHT_STD, device)
    out["b_qkv"] = _draw(g, (3 * d,), BIAS_SCALE, device)
    out["W_o"] = _draw(g, (d, d), WEIGHT_STD, device)
    out["b_o"] = _draw(g, (d,), BIAS_SCALE, device)
    out["W_up"] = _draw(g, (d, F), WEIGHT_STD, device)
    out["b_up"] = _draw(g, (F,), BIAS_SCALE, device)
    out["W_down"] = _draw(g, (F, d), WEIGHT_STD, device)
    out["b_down"] = _draw(g, (d,), BIAS_SCALE, device)
    for k in ("ln1", "ln2"):
        out[k + "_g"] = (1.0 + WEIGHT_STD * torch.randn(d, generator=g, device=device)).to(torch.bfloat16)
        out[k + "_b"] = _draw(g, (d,), WEIGHT_STD, device)
    out["dY"] = _draw(g, (N, d), 1.0, device)
    return out


def decode_attn_inputs(B, d, n_heads, n_kv, head_dim, L_max, bias=True, seed=0, device="cpu"):
    """One decode step of a grouped-query attention block, drawn in this order:
    x (B, d) ~ N(0,1); W_qkv (d, (n_heads + 2 n_kv) head_dim) laid out
    [Q heads | K heads | V heads] and W_o (n_heads head_dim, d) ~ N(0, 0.02);
    biases 0.01 N(0,1); the cached keys and values of the earlier tokens
    K, V [n_kv][B][L_max][head_dim] ~ N(0, (0.02 sqrt(d))^2) -- the spread of
    x W_k for such x and W -- rounded to IEEE fp16, the cache's storage type."""
    g = make_generator(seed, device)
    nq, nk = n_heads * head_dim, n_kv * head_dim
    out = {"x": _draw(g, (B, d), 1.0, device), "W_qkv": _draw(g, (d, nq + 2 * nk), WEIGHT_STD, device)}
    out["b_qkv"] = _draw(g, (nq + 2 * nk,), BIAS_SCALE, device) if bias else None
    out["W_o"] = _draw(g, (nq, d), WEIGHT_STD, device)
    out["b_o"] = _draw(g, (d,), BIAS_SCALE, device) if bias else None
    kv_std = WEIGHT_STD * float(d) ** 0.5
    for k in ("K", "V"):
        out[k] = (kv_std * torch.randn(n_kv, B, L_max, head_dim, generator=g, device=device)).to(torch.float16)
    return out


def gqa_attn_inputs(N, d, n_heads, n_kv, head_dim, bias=True, dy=True, seed=0, device="cpu"):
    """Grouped-query attention block: Xn (N, d), W_qkv (d, (n_heads + 2 n_kv) head_dim)
    laid out [Q heads | K heads | V heads], b_qkv, W_o (n_heads head_dim, d), b_o, dY."""
    g = make_generator(seed, device)
    nq, nk = n_heads * head_dim, n_kv * head_dim
    out = {"X": _draw(g, (N, d), 1.0, device), "W_qkv": _draw(g, (d, nq + 2 * nk), WEIGHT_STD, device)}
    out["b_qkv"] = _draw(g, (nq + 2 * nk,), BIAS_SCALE, device) if bias else None
    out["W_o"] = _draw(g, (nq, d), WEIGHT_STD, device)
    out["b_o"] = _draw(g, (d,), BIAS_SCALE, device) if bias else None
    out["dY"] = _draw(g, (N, d), 1.0, device) if dy else None
    return out


def token_ids(N, V, zipf_s=1.1, seed=0):
    """Seeded token ids in [0, V): a Zipf-shaped frequency (rank r drawn with
    weight r^-s, ranks mapped to ids through a seeded permutation) so that a
    few ids repeat often, as in text.  int32."""
    g = make_generator(seed + 104729, "cpu")
    ranks = torch.arange(1, V + 1, dtype=torch.float64)
    w = ranks.pow(-zipf_s)
    r = torch.multinomial(w / w.sum(), N, replacement=True, generator=g)
    perm = torch.randperm(V, generator=g)
    return perm[r].to(torch.int32)


def embedding_inputs(N, V, h, seed=0, device="cpu"):
    """E (V, h) ~ N(0, 0.02) and dY (N, h) ~ N(0, 1), bf16, drawn in that order."""
    g = make_generator(seed, device)
    return {"E": _draw(g, (V, h), WEIGHT_STD, device), "dY": _draw(g, (N, h), 1.0, device)}


def decode_positions(B, lo, hi, seed=0):
    """Seeded cache positions, uniform on [lo, hi] (a ragged length mix), int32."""
    g = make_generator(seed + 7919, "cpu")
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int32)


def f16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw IEEE fp16 bit patterns of a (CPU) fp16 tensor as a uint16 array."""
    assert t.dtype == torch.float16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a (CPU) bf16 tensor as a uint16 array."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
