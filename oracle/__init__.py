"""fp64 CPU oracle for the fused linear cross-entropy (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  It does not import the library.
"""
from .flce_oracle import (  # noqa: F401
    STATUS_OK, STATUS_TARGET_OUT_OF_RANGE, backward, dhidden_rows, dweight_rows,
    forward, forward_rows, grad_logits, logits, lse_all, relative_frobenius,
    token_weights, widen,
)
