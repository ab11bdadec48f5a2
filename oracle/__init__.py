"""fp64 CPU oracle for block-sparse gated causal prefill attention.

TEST INFRASTRUCTURE ONLY: imported by the tests, ``__graft_entry__.smoke()``
and the CPU-baseline legs of ``bench.py``; never by the product package.
"""
from . import bsfa_oracle, guard  # noqa: F401
