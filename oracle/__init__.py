"""fp64 CPU oracle for the Megatron tensor-parallel transformer block.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
executes this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It
shares no code with the CUDA library (``megatron_tensor_transformer_shard_gb300``)
and imports nothing from it; both sides only consume the same seeded input
bits.

Everything here is the plain definition of what the method computes, in
float64 on bf16-rounded inputs, written out step by step so that it can be
checked against the pages by eye.  Library matmuls (``@``) serve as steps; no
blocking, fusion or reordering beyond what the definitions state.

Parity status: every function is pinned by tests/test_oracle_*.py against
values the pages print, closed forms, invariants or brute-force finite
differences; there is no "parity unpinned" function.
"""

from .tp_oracle import *  # noqa: F401,F403
from .tp_gqa_decode import *  # noqa: F401,F403
from .tp_embedding import *  # noqa: F401,F403
