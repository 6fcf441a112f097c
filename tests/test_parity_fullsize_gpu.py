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
    """The fused call (automatic backward: kept logits from D = 1152 up, else the recompute), as
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
    dW_ref, db_ref = oracle.dweight_rows(hc, Wc, bc, tc, vrows.numpy(), ref["lse"], dloss=dlc, **kw)
    err = {"dhidden": oracle.relative_frobenius(dh_g, dh_ref), "dweight": oracle.relative_frobenius(dW_g, dW_ref)}
    if db_g is not None:
        err["dbias"] = oracle.relative_frobenius(db_g, db_ref)
    print(f"{name} {entry}{' compact' if compact else ''}: relative Frobenius errors "
          + ", ".join(f"{k} {v:.2e}" for k, v in err.items()))
    assert all(v <= TOL_GRAD for v in err.values()), err
    if w.hidden_dtype == torch.float32:
        # dweight = G^T h reads h's leading bf16 term only: G itself is rounded to bf16, so the
        # error is that of two bf16 roundings (RMS about 2^-9 / sqrt(3) each), far inside 1e-2
        assert err["dweight"] <= 5e-3, err


def test_long_context_131k_tokens():
    """A step of 131072 tokens (8 x the Qwen3-8B-like batch; the pages' long-context range) through
    the fused call (kept logits, 26 token chunks) and the separate calls (recompute, 38 vocabulary
    chunks).  The oracle cannot sweep all tokens in fp64 here, so it checks sampled tokens: lse,
    entropy and per-token loss of 256 tokens, dhidden of 64.  dweight and dbias are checked by what
    holds at any size: without a soft cap every row of G sums to zero, so their sums over the
    vocabulary vanish up to bf16 rounding (about 2^-9 of their norm); and the two algorithms agree."""
    import linear_cross_entropy_tmem_gb300 as F
    w = WORKLOADS["qwen8b"].scaled(name="Qwen3-8B-like N131072", n_tokens=131072, reduction="none", bias=True)
    h, W, b, t, dloss = make_inputs(w, "cuda")
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)
    fwd, grads = F.flce_forward_backward(h, W, t, dloss, b, entropy=True, **kw)
    torch.cuda.synchronize()
    assert F.flce_read_device_status(fwd.workspace) == 0
    sep = run_gpu(h, W, b, t, dloss, **kw)
    assert sep["status"] == 0
    tc = t.cpu().numpy()
    nv = int(((tc != -100) & (tc >= 0) & (tc < w.vocab)).sum())
    for f in (fwd, sep["fwd"]):
        assert int(f.n_valid) == nv and 0 <= int(f.correct) <= nv
    g = torch.Generator().manual_seed(77)
    rows = torch.randperm(w.n_tokens, generator=g)[:256].sort().values
    hc, Wc, bc, dlc = h.cpu(), W.cpu(), b.cpu(), dloss.cpu()
    ref = oracle.forward_rows(hc, Wc, bc, t.cpu(), rows.numpy(), **kw)
    for f in (fwd, sep["fwd"]):
        np.testing.assert_allclose(f.lse[rows.cuda()].double().cpu().numpy(), ref["lse"], atol=TOL_LSE, rtol=0)
        np.testing.assert_allclose(f.entropy[rows.cuda()].double().cpu().numpy(), ref["entropy"], atol=TOL_ENT,
                                   rtol=0)
        np.testing.assert_allclose(f.loss[rows.cuda()].double().cpu().numpy(), ref["loss"], atol=TOL_LOSS, rtol=0)
    dh_ref = oracle.dhidden_rows(hc, Wc, bc, t.cpu(), rows[:64].numpy(), n_valid=nv, dloss=dlc, **kw)
    for dh, dW, db in (grads, sep["bwd"]):
        assert oracle.relative_frobenius(dh[rows[:64].cuda()].cpu(), dh_ref) <= TOL_GRAD
        dWd = dW.double()
        assert torch.isfinite(dWd).all() and float(dWd.norm()) > 0
        assert float(dWd.sum(dim=0).norm()) <= 0.01 * float(dWd.norm())
        assert abs(float(db.double().sum())) <= 0.01 * float(db.double().norm())
    assert oracle.relative_frobenius(grads[1].cpu(), sep["bwd"][1].cpu()) <= TOL_GRAD
    assert oracle.relative_frobenius(grads[2].cpu(), sep["bwd"][2].cpu()) <= TOL_GRAD


@pytest.mark.parametrize("N,D,V,softcap", [(600, 1024, (1 << 20) + 3, 0.0), (1100, 1280, 1 << 20, 0.0),
                                           (2048, 8192, 32000, 30.0)],
                         ids=["V1M-ragged-recompute", "V1M-keep-logits", "D8192-softcap"])
def test_extreme_shapes(N, D, V, softcap):
    """Very large shapes: a vocabulary of 2^20 (+3: ragged tiles everywhere) through the recompute
    and the token-chunked backward, and an 8192-wide hidden state with a soft cap.  The oracle
    checks 128 sampled tokens (lse, entropy, per-token loss) and dhidden on 32 of them; dweight and
    dbias are checked by what holds at any size (without a soft cap each row of G sums to zero, so
    their sums over the vocabulary vanish up to bf16 rounding) and by the fused call agreeing with
    flce_forward + flce_backward, a different algorithm from D = 1152 up."""
    import linear_cross_entropy_tmem_gb300 as F
    from tests.parity import run_gpu
    w = WORKLOADS["tiny"].scaled(name=f"extreme N{N} D{D} V{V}", n_tokens=N, hidden=D, vocab=V,
                                 sigma_w=0.5 / D ** 0.5, softcap=softcap, bias=True, reduction="none", seed=41)
    h, W, b, t, dloss = make_inputs(w, "cuda")
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)
    fwd, grads = F.flce_forward_backward(h, W, t, dloss, b, entropy=True, **kw)
    torch.cuda.synchronize()
    assert F.flce_read_device_status(fwd.workspace) == 0
    sep = run_gpu(h, W, b, t, dloss, **kw)
    assert sep["status"] == 0
    tc = t.cpu().numpy()
    nv = int(((tc != -100) & (tc >= 0) & (tc < V)).sum())
    g = torch.Generator().manual_seed(5)
    rows = torch.randperm(N, generator=g)[:128].sort().values
    hc, Wc, bc, dlc = h.cpu(), W.cpu(), b.cpu(), dloss.cpu()
    ref = oracle.forward_rows(hc, Wc, bc, t.cpu(), rows.numpy(), **kw)
    for f in (fwd, sep["fwd"]):
        assert int(f.n_valid) == nv
        np.testing.assert_allclose(f.lse[rows.cuda()].double().cpu().numpy(), ref["lse"], atol=TOL_LSE, rtol=0)
        np.testing.assert_allclose(f.entropy[rows.cuda()].double().cpu().numpy(), ref["entropy"], atol=TOL_ENT,
                                   rtol=0)
        np.testing.assert_allclose(f.loss[rows.cuda()].double().cpu().numpy(), ref["loss"], atol=TOL_LOSS, rtol=0)
    dh_ref = oracle.dhidden_rows(hc, Wc, bc, t.cpu(), rows[:32].numpy(), n_valid=nv, dloss=dlc, **kw)
    for dh, dW, db in (grads, sep["bwd"]):
        assert oracle.relative_frobenius(dh[rows[:32].cuda()].cpu(), dh_ref) <= TOL_GRAD
        dWd = dW.double()
        assert torch.isfinite(dWd).all() and float(dWd.norm()) > 0
        if softcap == 0.0:
            assert float(dWd.sum(dim=0).norm()) <= 0.01 * float(dWd.norm())
            assert abs(float(db.double().sum())) <= 0.01 * float(db.double().norm())
    for a, c in zip(grads[1:], sep["bwd"][1:]):  # on the device: dweight is up to 2 GB here
        assert float((a.double() - c.double()).norm()) <= TOL_GRAD * float(c.double().norm())
