"""CPU oracle of the block-scaled fused MoE layer (FP64, numpy).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the product path.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
in ``tests/test_oracle_*.py`` (format tables against independent decoders
and closed forms, the quantisation rule against hand cases and error
bounds, the sort against brute force and permutation invariants, the layer
against a brute-force scalar evaluation on tiny shapes, the dense-MLP
special case, zero-weight and linearity invariants).
"""
from . import mx_formats, moe  # noqa: F401
