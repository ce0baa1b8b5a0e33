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


GUARD_BYTE = 0xA5


class Guarded:
    """A device buffer with `pad` guard bytes before and after it, all filled
    with GUARD_BYTE before the call under test.  ``.t`` is the tensor the
    kernel may write (shape, dtype as given; the first byte 256-aligned);
    ``.check(name)`` asserts that neither guard changed, i.e. nothing was
    written outside the tensor.  ``fill`` sets the tensor's own initial bytes
    (default: the guard pattern too, so unwritten elements stay recognisable)."""

    def __init__(self, shape, dtype, pad=4096, fill=None):
        import math
        shape = tuple(int(s) for s in (shape if isinstance(shape, (tuple, list)) else (shape,)))
        itemsize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = math.prod(shape) * itemsize
        self.pad = pad
        self.buf = torch.full((pad + self.nbytes + pad,), GUARD_BYTE, dtype=torch.uint8, device="cuda")
        self.t = self.buf[pad:pad + self.nbytes].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def check(self, name):
        torch.cuda.synchronize()
        head = self.buf[:self.pad].cpu().numpy()
        tail = self.buf[self.pad + self.nbytes:].cpu().numpy()
        bad_h = np.nonzero(head != GUARD_BYTE)[0]
        bad_t = np.nonzero(tail != GUARD_BYTE)[0]
        assert bad_h.size == 0, f"{name}: {bad_h.size} guard bytes changed before the buffer (first at -{self.pad - bad_h[0]})"
        assert bad_t.size == 0, f"{name}: {bad_t.size} guard bytes changed after the buffer (first at +{bad_t[0]})"


def guarded_ws(nbytes, pad=4096):
    """Workspace of exactly `nbytes` (at least 16) between guard regions."""
    return Guarded((max(int(nbytes), 16),), torch.uint8, pad=pad)
