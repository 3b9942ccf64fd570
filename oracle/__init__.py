"""CPU oracle (float64) for causal multi-head self-attention, forward and backward.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
benchmark's CPU-baseline leg, never by the product path. It shares no code with
the CUDA kernels or their host library.

Parity pins: every function here is pinned by tests that do not re-type its
formulas (hand-worked example, closed forms, invariants, finite differences,
library cross-checks); see tests/test_oracle_pins.py.
"""
from .attention import (forward, backward, head_forward, head_backward,  # noqa: F401
                        head_dpreatt_jacobian, split_heads, row_stat_D)
from .layer import linear, block_forward  # noqa: F401
