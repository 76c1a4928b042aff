"""CPU oracle (float64) for the token-choice MoE layer: test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it; the CUDA path never does.
"""
from . import moe_oracle  # noqa: F401
