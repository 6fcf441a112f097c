"""Fused linear cross-entropy for GB300 (sm_103a): a thin binding over ``libflce.so``.

The library computes the next-token cross-entropy of ``hidden @ weight.T`` (with
an optional bias, logit scale and soft cap), forward and backward, without
materialising the (tokens x vocab) logits.  See ``include/flce.h``.
"""
from .api import (  # noqa: F401
    ForwardResult, LinearCrossEntropy, flce_backward, flce_forward, flce_forward_backward, flce_read_device_status,
    flce_status_string, flce_workspace_size, linear_cross_entropy, make_problem, scale_gradient,
)
