"""flce_forward_noalloc: the forward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: a plugin inside a host application that
owns the device-memory budget and gives its plugins no allocator, or
latency-critical code that cannot accept cudaMalloc's implicit device
synchronisation.  This entry point keeps its scratch in a static device array
inside the library instead of a caller workspace.

The GPU test calls it several times in a row through the C ABI, on different
problems, so that each call starts from the previous call's leftover scratch:
bf16 and fp32 hidden states, bias, scale and soft cap, every reduction, and a
problem whose forward workspace is just under the array's size.  Each result
must equal the regular flce_forward's bit for bit (the same kernels and plan on
the same inputs), and the first is also compared with the fp64 oracle at the
parity tolerances.  This file is collected last, so that a run stopping at its
first failure has already run every other test.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import oracle
from linear_cross_entropy_tmem_gb300 import binding as B
from linear_cross_entropy_tmem_gb300.synthetic import Workload, make_inputs
from tests.parity import compare_forward

NOALLOC_BYTES = 32 << 20  # FLCE_NOALLOC_SCRATCH_BYTES


def _p(t):
    return None if t is None or t.numel() == 0 else ctypes.c_void_p(t.data_ptr())


def _problem(w, h, b):
    import linear_cross_entropy_tmem_gb300.api as api
    return api.make_problem(h.shape[0], h.shape[1], w.vocab, hidden_dtype=h.dtype,
                            bias_dtype=b.dtype if b is not None else torch.bfloat16,
                            logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)


def _noalloc_forward(lib, w, h, W, b, t):
    N = h.shape[0]
    prob = _problem(w, h, b)
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


def _largest_tokens_below_limit(V, D):
    """The largest N (a multiple of 64) whose forward workspace still fits the static array."""
    import linear_cross_entropy_tmem_gb300.api as api
    lo, hi = 64, 1 << 20
    while hi - lo > 64:
        mid = (lo + hi) // 2 // 64 * 64
        if api.flce_workspace_size(api.make_problem(mid, D, V), False) <= NOALLOC_BYTES:
            lo = mid
        else:
            hi = mid
    return lo


PROBLEMS = [
    Workload("noalloc-a bf16 bias s0.8 c6 mean", 1000, 256, 5000, sigma_w=0.2, bias=True, logit_scale=0.8,
             softcap=6.0, seed=21),
    Workload("noalloc-b bf16 none", 300, 128, 3000, sigma_w=0.3, reduction="none", seed=22),
    Workload("noalloc-c fp32-h bias-f32 s0.0625 c30 sum", 700, 192, 4100, sigma_w=0.3,
             hidden_dtype=torch.float32, bias=True, logit_scale=0.0625,
             softcap=30.0, reduction="sum", seed=23),
]


@pytest.mark.gpu
def test_noalloc_forward_equals_forward_bitwise_on_calls_in_a_row(lib):
    """Calls in a row on different problems (each starting from the last one's scratch) give exactly
    flce_forward's results; the first also matches the oracle."""
    import linear_cross_entropy_tmem_gb300 as F
    V, D = 16384, 64
    n_big = _largest_tokens_below_limit(V, D)
    big = Workload("noalloc-d bf16 at the scratch limit", n_big, D, V, sigma_w=0.1, seed=24)
    import linear_cross_entropy_tmem_gb300.api as api
    need = api.flce_workspace_size(api.make_problem(n_big, D, V), False)
    assert NOALLOC_BYTES - (4 << 20) < need <= NOALLOC_BYTES, need
    for i, w in enumerate(PROBLEMS + [big, PROBLEMS[0]]):
        h, W, b, t, _ = [x.cuda() if x is not None else None for x in make_inputs(w, "cpu")]
        if "bias-f32" in w.name:
            b = b.float()
        got = _noalloc_forward(lib, w, h, W, b, t)
        ref = F.flce_forward(h, W, t, b, logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction,
                             entropy=True)
        torch.cuda.synchronize()
        assert F.flce_read_device_status(ref.workspace) == 0
        for k in ("lse", "entropy", "entropy_sum", "correct", "n_valid"):
            assert torch.equal(got[k], getattr(ref, k).reshape(got[k].shape)), (w.name, k)
        assert torch.equal(got["loss"], ref.loss.reshape(got["loss"].shape)), (w.name, "loss")
        if i == 0:
            hc, Wc, bc, tc = (x.cpu() if x is not None else None for x in (h, W, b, t))
            kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)
            res = F.ForwardResult(*[got[k] if k in got else None for k in F.ForwardResult._fields])
            compare_forward(res, oracle.forward(hc, Wc, bc, tc, **kw), reduction=w.reduction,
                            z=oracle.logits(hc, Wc, bc, logit_scale=w.logit_scale, softcap=w.softcap),
                            t=tc.numpy())


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
