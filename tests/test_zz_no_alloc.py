"""flce_forward_noalloc: the forward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (a plugin in a host application that owns
the device-memory budget, or latency-critical code that cannot accept
cudaMalloc's implicit synchronisation).  This entry point keeps its scratch in
a static device array inside the library instead of a caller workspace.  The
GPU test calls it twice in a row through the C ABI, on two different problems so
that the second call starts from the first call's leftover scratch, and checks
each result against the regular flce_forward within the parity tolerances.
This file is collected last so that a run stopping at its first failure has
already run every other test.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

from linear_cross_entropy_tmem_gb300 import binding as B
from linear_cross_entropy_tmem_gb300.synthetic import Workload, make_inputs
from tests.parity import TOL_ENT, TOL_LOSS, TOL_LSE

NOALLOC_BYTES = 32 << 20  # FLCE_NOALLOC_SCRATCH_BYTES


def _p(t):
    return None if t is None or t.numel() == 0 else ctypes.c_void_p(t.data_ptr())


def _noalloc_forward(lib, w, h, W, b, t):
    import linear_cross_entropy_tmem_gb300.api as api
    N = h.shape[0]
    prob = api.make_problem(N, h.shape[1], W.shape[0], hidden_dtype=h.dtype,
                            bias_dtype=b.dtype if b is not None else torch.bfloat16,
                            logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)
    f32 = dict(dtype=torch.float32, device=h.device)
    out = {
        "loss": torch.full((N if w.reduction == "none" else 1,), float("nan"), **f32),
        "lse": torch.full((N,), float("nan"), **f32),
        "entropy": torch.full((N,), float("nan"), **f32),
        "correct": torch.full((1,), -1, dtype=torch.int64, device=h.device),
        "n_valid": torch.full((1,), -1, dtype=torch.int64, device=h.device),
        "entropy_sum": torch.full((1,), float("nan"), **f32),
    }
    st = lib.flce_forward_noalloc(ctypes.byref(prob), _p(h), _p(W), _p(b), _p(t), _p(out["loss"]),
                                  _p(out["lse"]), _p(out["entropy"]), _p(out["correct"]), _p(out["n_valid"]),
                                  _p(out["entropy_sum"]),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    B.check(st, "flce_forward_noalloc")
    torch.cuda.synchronize()
    return out


@pytest.mark.gpu
def test_noalloc_forward_matches_forward_on_two_calls_in_a_row(lib):
    import linear_cross_entropy_tmem_gb300 as F
    problems = [
        Workload("noalloc-a", 1000, 256, 5000, sigma_w=0.2, bias=True, logit_scale=0.8, softcap=6.0, seed=21),
        Workload("noalloc-b", 300, 128, 3000, sigma_w=0.3, reduction="none", seed=22),
    ]
    for w in problems:
        h, W, b, t, _ = [x.cuda() if x is not None else None for x in make_inputs(w, "cpu")]
        ref = F.flce_forward(h, W, t, b, logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction,
                             entropy=True)
        got = _noalloc_forward(lib, w, h, W, b, t)
        assert torch.allclose(got["lse"], ref.lse, atol=TOL_LSE, rtol=0)
        assert torch.allclose(got["entropy"], ref.entropy, atol=TOL_ENT, rtol=0)
        n = max(1, int(ref.n_valid))
        loss_tol = TOL_LOSS * (n if w.reduction == "sum" else 1)
        assert torch.allclose(got["loss"].reshape(ref.loss.shape), ref.loss, atol=loss_tol, rtol=0)
        assert int(got["correct"]) == int(ref.correct)
        assert int(got["n_valid"]) == int(ref.n_valid)
        assert abs(float(got["entropy_sum"]) - float(ref.entropy_sum)) <= TOL_ENT * n


def test_noalloc_rejects_problems_beyond_the_static_scratch(lib):
    """A forward whose workspace exceeds the static array is refused before any launch."""
    import linear_cross_entropy_tmem_gb300.api as api
    big = api.make_problem(400000, 4096, 151936)
    assert api.flce_workspace_size(big, False) > NOALLOC_BYTES
    fake = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(10)]
    st = lib.flce_forward_noalloc(ctypes.byref(big), *fake, None)
    assert st == B.FLCE_ERR_WORKSPACE_TOO_SMALL
    bad = api.make_problem(16, 130, 100)  # D not a multiple of 8
    assert lib.flce_forward_noalloc(ctypes.byref(bad), *fake, None) == B.FLCE_ERR_MISALIGNED
