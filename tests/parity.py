"""Shared helpers of the GPU parity tests: run the library and the oracle on the
same seeded inputs and compare with the tolerances of the target:

* integers (correct count, n_valid) bit-exact, except that positions whose two
  largest logits are within 1e-3 may flip (the count must lie in the range
  those positions allow);
* per-token loss and lse within 2e-3 absolute, entropy within 5e-3 absolute;
  scalar sums within the per-token bound times the number of valid tokens
  (a sum of n errors each within e is within n e);
* dhidden, dweight, dbias within 1e-2 relative Frobenius error.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL_LSE = 2e-3
TOL_LOSS = 2e-3
TOL_ENT = 5e-3
TOL_GRAD = 1e-2
NEAR_TIE = 1e-3


def run_gpu(h, W, b, t, dloss, *, logit_scale, softcap, reduction, ignore_index=-100, backward=True,
            num_items_in_batch=0.0, compact=False, fp32_full=False):
    import linear_cross_entropy_tmem_gb300 as F
    kw = dict(logit_scale=logit_scale, softcap=softcap, ignore_index=ignore_index, reduction=reduction,
              num_items_in_batch=num_items_in_batch, compact=compact, fp32_full=fp32_full)
    f = F.flce_forward(h, W, t, b, entropy=True, **kw)
    out = {"fwd": f}
    if backward:
        out["bwd"] = F.flce_backward(h, W, t, f.lse, f.n_valid, dloss, b, **kw)
    torch.cuda.synchronize()
    out["status"] = F.flce_read_device_status(f.workspace)
    return out


def launch_kinds(fn, cap=256):
    """Run fn() with the library's launch log on; return the kinds (binding.LAUNCH_KINDS names) of the
    kernels it launched, in order."""
    import ctypes

    from linear_cross_entropy_tmem_gb300 import binding as B
    lib = B.load()
    recs = (B.FlceLaunchRecord * cap)()
    events = []
    for i in range(cap):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()  # torch creates the CUDA event on its first record
        e1.record()
        events.append((e0, e1))
        recs[i].begin_event = ctypes.c_void_p(e0.cuda_event)
        recs[i].end_event = ctypes.c_void_p(e1.cuda_event)
    count = ctypes.c_int32(0)
    torch.cuda.synchronize()
    B.check(lib.flce_testing_set_launch_log(recs, cap, ctypes.byref(count)), "launch log")
    try:
        out = fn()
        torch.cuda.synchronize()
    finally:
        B.check(lib.flce_testing_set_launch_log(None, 0, None), "launch log")
    return out, [B.LAUNCH_KINDS[recs[i].kind] for i in range(count.value)]


def correct_bounds(z: np.ndarray, t: np.ndarray, valid: np.ndarray, argmax: np.ndarray):
    """Range of correct counts a kernel may report when near-ties (gap < 1e-3) flip."""
    rows = np.arange(z.shape[0])
    zs = np.sort(z, axis=1)
    gap = zs[:, -1] - zs[:, -2] if z.shape[1] > 1 else np.full(z.shape[0], np.inf)
    near = valid & (gap < NEAR_TIE)
    ora_ok = valid & (argmax == t)
    zmax = zs[:, -1]
    tt = np.where(valid, t, 0)
    target_close = valid & (zmax - z[rows, tt] < NEAR_TIE)
    lo = int(ora_ok.sum()) - int((near & ora_ok).sum())
    hi = int(ora_ok.sum()) + int((near & ~ora_ok & target_close).sum())
    return lo, hi


def compare_forward(gpu_f, ref, *, reduction, z=None, t=None):
    lse = gpu_f.lse.double().cpu().numpy()
    np.testing.assert_allclose(lse, ref["lse"], atol=TOL_LSE, rtol=0, err_msg="lse")
    ent = gpu_f.entropy.double().cpu().numpy()
    np.testing.assert_allclose(ent, ref["entropy"], atol=TOL_ENT, rtol=0, err_msg="entropy")
    nv = int(gpu_f.n_valid.item())
    assert nv == ref["n_valid"], ("n_valid", nv, ref["n_valid"])
    if reduction == "none":
        np.testing.assert_allclose(gpu_f.loss.double().cpu().numpy(), ref["loss"], atol=TOL_LOSS, rtol=0,
                                   err_msg="per-token loss")
    elif reduction == "mean":
        assert abs(gpu_f.loss.item() - ref["loss"]) <= TOL_LOSS, ("mean loss", gpu_f.loss.item(), ref["loss"])
    else:
        assert abs(gpu_f.loss.item() - ref["loss"]) <= TOL_LOSS * max(1, nv), ("sum loss", gpu_f.loss.item(),
                                                                              ref["loss"])
    assert abs(gpu_f.entropy_sum.item() - ref["entropy_sum"]) <= TOL_ENT * max(1, nv), \
        ("entropy_sum", gpu_f.entropy_sum.item(), ref["entropy_sum"])
    c = int(gpu_f.correct.item())
    if z is not None:
        lo, hi = correct_bounds(z, t, ref["valid"], ref["argmax"])
        assert lo <= c <= hi, ("correct", c, lo, hi, ref["correct"])
    else:
        assert c == ref["correct"], ("correct", c, ref["correct"])


def compare_backward(gpu_b, ref):
    dh, dW, db = gpu_b
    for name, g, r in (("dhidden", dh, ref["dh"]), ("dweight", dW, ref["dW"]), ("dbias", db, ref["db"])):
        if r is None:
            assert g is None
            continue
        err = oracle.relative_frobenius(g, r)
        assert err <= TOL_GRAD, (name, err)


def oracle_forward_rowblocks(h, W, b, t, *, row_block=256, **kw):
    """The oracle's forward applied to consecutive groups of tokens (every output
    is per token; the scalar reductions are sums over the groups).  Inputs are
    widened to fp64 once so that each group only pays for its own logits."""
    hf = oracle.widen(h)
    Wf = oracle.widen(W)
    bf = None if b is None else oracle.widen(b)
    tt = np.asarray(t.cpu().numpy() if hasattr(t, "cpu") else t)
    red = kw.pop("reduction", "mean")
    parts = [oracle.forward(hf[r:r + row_block], Wf, bf, tt[r:r + row_block], reduction="none", **kw)
             for r in range(0, hf.shape[0], row_block)]
    out = {k: np.concatenate([p[k] for p in parts]) for k in ("loss_tok", "lse", "entropy", "argmax", "valid")}
    out["n_valid"] = int(sum(p["n_valid"] for p in parts))
    out["correct"] = int(sum(p["correct"] for p in parts))
    out["entropy_sum"] = float(sum(p["entropy_sum"] for p in parts))
    total = float(out["loss_tok"].sum())
    out["loss"] = {"sum": total, "mean": total / out["n_valid"] if out["n_valid"] else 0.0,
                   "none": out["loss_tok"]}[red]
    out["status"] = max(p["status"] for p in parts)
    return out


def near_tie_bounds_rowblocks(h, W, b, t, ref, *, row_block=256, logit_scale=1.0, softcap=0.0):
    """correct_bounds() over groups of tokens (only needed when the counts differ)."""
    hf = oracle.widen(h)
    Wf = oracle.widen(W)
    bf = None if b is None else oracle.widen(b)
    tt = np.asarray(t.cpu().numpy() if hasattr(t, "cpu") else t)
    lo = hi = 0
    for r in range(0, hf.shape[0], row_block):
        z = oracle.logits(hf[r:r + row_block], Wf, bf, logit_scale=logit_scale, softcap=softcap)
        a, c = correct_bounds(z, tt[r:r + row_block], ref["valid"][r:r + row_block], ref["argmax"][r:r + row_block])
        lo += a
        hi += c
    return lo, hi
