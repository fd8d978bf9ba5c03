"""CPU oracle for the top-k MoE FFN forward pass.

TEST INFRASTRUCTURE: only the tests, `__graft_entry__.smoke()` and the CPU-baseline /
reference legs of `bench.py` import this package.  The CUDA library never does.
"""
from . import moe_oracle
from .cases import Case, gapped_attempts

__all__ = ["moe_oracle", "Case", "gapped_attempts"]
