"""Shared helpers of the GPU parity tests: move seeded inputs to the device,
read results back as float64, and the parity criterion

    max |gpu - oracle| <= 1e-2 * max |oracle|      (per output tensor)

which is what bf16 inputs with fp32 accumulation are held to against an fp64
oracle on the same bf16-rounded inputs.  Bit-exact checks (packing) compare
raw uint16 bit patterns.
"""

import numpy as np
import torch

import oracle as O
from megatron_tensor_transformer_shard_gb300 import inputs as I

TOL = 1e-2


def f64(t: torch.Tensor) -> np.ndarray:
    """bf16 or fp32 tensor (any device) -> float64 numpy."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return O.bf16_to_f64(I.bits(t)).reshape(tuple(t.shape))
    return t.double().numpy()


def rel_err(gpu, ref) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), "non-finite GPU output"
    return float(np.abs(gpu - ref).max() / max(np.abs(ref).max(), 1e-30))


def assert_close(name, gpu, ref, tol=TOL):
    e = rel_err(gpu, ref)
    assert e <= tol, f"{name}: max|gpu-oracle| / max|oracle| = {e:.3e} > {tol}"
    return e


def empty_bf16(*shape):
    return torch.empty(*shape, dtype=torch.bfloat16, device="cuda")


def empty_f32(*shape):
    return torch.empty(*shape, dtype=torch.float32, device="cuda")


def ws_bytes(n):
    return torch.empty(max(int(n), 16), dtype=torch.uint8, device="cuda")
