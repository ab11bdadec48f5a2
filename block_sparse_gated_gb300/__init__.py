"""GB300-native block-sparse gated causal prefill attention (BSFA form).

The compute path is the C-ABI library ``libbsfa.so`` built from ``csrc/`` for
sm_103a; this package only marshals torch tensors into its calls.  Importing
the package does not load the library; the first call does, and fails loudly
if it has not been built.
"""
from .api import (  # noqa: F401
    GATE_LAMBDA,
    GATE_NONE,
    GATE_THRESHOLD,
    BsfaError,
    bitmap_shape,
    calibrate,
    prefill,
)
