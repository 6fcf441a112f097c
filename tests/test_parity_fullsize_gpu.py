"""GPU parity at the five benchmark sizes, in the launch configuration bench.py
times (the fused call with its automatic backward, same planner, same seeded
device draws), plus flce_forward + flce_backward and valid-token compaction.

Per-token outputs are compared on every token against the oracle's forward run
over groups of tokens; the scalar outputs against its sums.  Gradients are
compared on sampled rows: 64 token rows of dhidden (each needs only its own
logits) and 64 vocabulary rows of dweight / dbias (computed from the oracle's
own full-vocabulary lse of every token)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from linear_cross_entropy_tmem_gb300.synthetic import WORKLOADS, make_inputs
from tests.parity import (TOL_ENT, TOL_GRAD, TOL_LOSS, TOL_LSE, near_tie_bounds_rowblocks,
                          oracle_forward_rowblocks, run_gpu)

pytestmark = [pytest.mark.gpu, pytest.mark.fullsize]


def _run(h, W, b, t, dloss, entry, compact, kw):
    """The fused call (automatic backward: kept logits from D = 1024 up, else the recompute), as
    bench.py times it, or flce_forward followed by flce_backward."""
    import linear_cross_entropy_tmem_gb300 as F
    if entry == "separate":
        gpu = run_gpu(h, W, b, t, dloss, compact=compact, **kw)
        return gpu["status"], gpu["fwd"], gpu["bwd"]
    fwd, grads = F.flce_forward_backward(h, W, t, dloss, b, entropy=True, compact=compact, **kw)
    torch.cuda.synchronize()
    return F.flce_read_device_status(fwd.workspace), fwd, grads


@pytest.mark.parametrize("name,compact,entry", [
    ("tiny", False, "fused"), ("chunk", False, "fused"), ("commandr", False, "fused"), ("gemma", False, "fused"),
    ("qwen8b", False, "fused"), ("qwen8b", False, "separate"), ("commandr", True, "fused")],
    ids=["tiny", "chunk", "commandr-keep-logits", "gemma", "qwen8b-keep-logits", "qwen8b-separate",
         "commandr-compact"])
def test_parity_full_size(name, compact, entry):
    w = WORKLOADS[name]
    h, W, b, t, dloss = make_inputs(w, "cuda")
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)
    status, f, (dh, dW, db) = _run(h, W, b, t, dloss, entry, compact, kw)
    assert status == 0
    g = torch.Generator().manual_seed(1234)
    rows = torch.randperm(w.n_tokens, generator=g)[:64].sort().values
    vrows = torch.randperm(w.vocab, generator=g)[:64].sort().values
    # the GPU results we compare, moved to the host
    lse_g, ent_g = f.lse.cpu().double().numpy(), f.entropy.cpu().double().numpy()
    loss_g = f.loss.cpu().double().numpy()
    dh_g = dh[rows.cuda()].cpu()
    dW_g = dW[vrows.cuda()].cpu()
    db_g = db[vrows.cuda()].cpu() if db is not None else None
    hc, Wc, tc, dlc = h.cpu(), W.cpu(), t.cpu(), dloss.cpu()
    bc = b.cpu() if b is not None else None
    del h, W, b, t, dloss, dh, dW, db
    torch.cuda.empty_cache()

    ref = oracle_forward_rowblocks(hc, Wc, bc, tc, **kw)
    v = ref["valid"] if compact else np.ones_like(ref["valid"])
    np.testing.assert_allclose(lse_g[v], ref["lse"][v], atol=TOL_LSE, rtol=0)
    np.testing.assert_allclose(ent_g[v], ref["entropy"][v], atol=TOL_ENT, rtol=0)
    if compact:  # ignored tokens are not computed: lse = entropy = 0
        assert np.all(lse_g[~v] == 0.0) and np.all(ent_g[~v] == 0.0)
    nv = ref["n_valid"]
    assert int(f.n_valid) == nv
    if w.reduction == "none":
        np.testing.assert_allclose(loss_g, ref["loss"], atol=TOL_LOSS, rtol=0)
    else:
        tol = TOL_LOSS * (nv if w.reduction == "sum" else 1)
        assert abs(float(loss_g.reshape(-1)[0]) - ref["loss"]) <= tol
    assert abs(float(f.entropy_sum) - ref["entropy_sum"]) <= TOL_ENT * max(1, nv)
    c = int(f.correct)
    if c != ref["correct"]:
        lo, hi = near_tie_bounds_rowblocks(hc, Wc, bc, tc, ref, logit_scale=w.logit_scale, softcap=w.softcap)
        assert lo <= c <= hi, (c, lo, hi)

    dh_ref = oracle.dhidden_rows(hc, Wc, bc, tc, rows.numpy(), n_valid=nv, dloss=dlc, **kw)
    assert oracle.relative_frobenius(dh_g, dh_ref) <= TOL_GRAD
    dW_ref, db_ref = oracle.dweight_rows(hc, Wc, bc, tc, vrows.numpy(), ref["lse"], dloss=dlc, **kw)
    assert oracle.relative_frobenius(dW_g, dW_ref) <= TOL_GRAD
    if db_g is not None:
        assert oracle.relative_frobenius(db_g, db_ref) <= TOL_GRAD
