"""Randomised GPU parity: seeded draws over shapes (ragged N, D, V), dtypes, bias, scale, soft
cap, reduction, ignore patterns, num_items_in_batch, compaction, the fused call's backward, the GEMM
kernel and the chunking knobs, each compared with the fp64 oracle element by element.  The draws are
reproducible from the seed in the test id."""
from __future__ import annotations

import random

import numpy as np
import pytest
import torch

import oracle
from linear_cross_entropy_tmem_gb300.synthetic import Workload, make_inputs
from tests.parity import TOL_ENT, TOL_GRAD, TOL_LOSS, TOL_LSE, correct_bounds, run_gpu

pytestmark = pytest.mark.gpu


def _draw(seed: int):
    r = random.Random(seed)
    fp32_h = r.random() < 0.3
    case = dict(
        N=r.choice([1, 7, 64, 129, 255, 256, 300, 511, 700]),
        D=8 * r.randint(1, 160) if r.random() < 0.8 else r.choice([1024, 1032, 1280]),
        V=r.choice([1, 5, 255, 256, 257, 1000, 2049, 4999]),
        bias=r.random() < 0.5, bias_f32=r.random() < 0.3, scale=r.choice([1.0, 0.5, 1.7]),
        softcap=r.choice([0.0, 0.0, 4.0, 30.0]), reduction=r.choice(["mean", "sum", "none"]),
        ignore_every=r.choice([0, 3, 17]), items=r.choice([0.0, 0.0, 123.0]),
        fp32_h=fp32_h, fp32_w=fp32_h and r.random() < 0.5, full=r.random() < 0.3,
        compact=r.random() < 0.3, entry=r.choice(["separate", "fused-auto", "fused-recompute", "fused-keep"]),
        mode=r.choice([0, 1, 2]), chunk_cols=r.choice([0, 0, 512]), ksplit=r.choice([0, 0, 2, 5]),
        token_chunk=r.choice([0, 256]), sigma=r.choice([0.05, 0.2, 0.6]),
    )
    if case["reduction"] != "mean":
        case["items"] = 0.0
    return case


@pytest.fixture(autouse=True)
def _reset_knobs():
    yield
    from linear_cross_entropy_tmem_gb300.api import testing_set_gemm_mode, testing_set_token_chunk, testing_set_tuning
    testing_set_tuning(0, 0)
    testing_set_gemm_mode(0)
    testing_set_token_chunk(0)


@pytest.mark.parametrize("seed", range(256))
def test_random_case_matches_oracle(seed):
    import linear_cross_entropy_tmem_gb300 as F
    from linear_cross_entropy_tmem_gb300.api import testing_set_gemm_mode, testing_set_token_chunk, testing_set_tuning
    c = _draw(seed)
    testing_set_gemm_mode(c["mode"])
    testing_set_tuning(c["chunk_cols"], c["ksplit"])
    testing_set_token_chunk(c["token_chunk"])
    w = Workload(f"fuzz{seed}", c["N"], c["D"], c["V"], sigma_w=c["sigma"] / max(1.0, c["D"] ** 0.5 / 8),
                 hidden_dtype=torch.float32 if c["fp32_h"] else torch.bfloat16, bias=c["bias"], logit_scale=c["scale"],
                 softcap=c["softcap"], reduction=c["reduction"], ignore_every=c["ignore_every"], seed=1000 + seed)
    h, W, b, t, dloss = make_inputs(w, "cpu")
    if b is not None and c["bias_f32"]:
        b = b.float()
    if c["fp32_w"]:
        g = torch.Generator().manual_seed(seed)
        W = (W.float() * (1.0 + 0.01 * torch.randn(W.shape, generator=g))).contiguous()
    dev = [x.cuda() if x is not None else None for x in (h, W, b, t, dloss)]
    kw = dict(logit_scale=c["scale"], softcap=c["softcap"], reduction=c["reduction"],
              num_items_in_batch=c["items"])
    if c["entry"] == "separate":
        gpu = run_gpu(*dev, compact=c["compact"], fp32_full=c["full"], **kw)
        status, f, grads = gpu["status"], gpu["fwd"], gpu["bwd"]
    else:
        bwd = {"fused-auto": "auto", "fused-recompute": "recompute", "fused-keep": "keep_logits"}[c["entry"]]
        f, grads = F.flce_forward_backward(dev[0], dev[1], dev[3], dev[4], dev[2], entropy=True, bwd=bwd,
                                           compact=c["compact"], fp32_full=c["full"], **kw)
        torch.cuda.synchronize()
        status = F.flce_read_device_status(f.workspace)
    assert status == 0, (c, status)
    ref_f = oracle.forward(h, W, b, t, **kw)
    ref_b = oracle.backward(h, W, b, t, dloss=dloss, **kw)
    valid = ref_f["valid"]
    rows = valid if c["compact"] else np.ones_like(valid)  # compaction leaves ignored tokens at 0
    lse, ent = f.lse.double().cpu().numpy(), f.entropy.double().cpu().numpy()
    np.testing.assert_allclose(lse[rows], ref_f["lse"][rows], atol=TOL_LSE, rtol=0, err_msg=str(c))
    np.testing.assert_allclose(ent[rows], ref_f["entropy"][rows], atol=TOL_ENT, rtol=0, err_msg=str(c))
    if c["compact"]:
        assert np.all(lse[~valid] == 0) and np.all(ent[~valid] == 0), c
    nv = int(f.n_valid)
    assert nv == ref_f["n_valid"], c
    if c["reduction"] == "none":
        np.testing.assert_allclose(f.loss.double().cpu().numpy(), ref_f["loss"], atol=TOL_LOSS, rtol=0,
                                   err_msg=str(c))
    else:
        tol = TOL_LOSS * (max(1, nv) if c["reduction"] == "sum" else 1)
        assert abs(float(f.loss) - ref_f["loss"]) <= tol, (c, float(f.loss), ref_f["loss"])
    assert abs(float(f.entropy_sum) - ref_f["entropy_sum"]) <= TOL_ENT * max(1, nv), c
    z = oracle.logits(h, W, b, logit_scale=c["scale"], softcap=c["softcap"])
    lo, hi = correct_bounds(z, t.numpy(), valid, ref_f["argmax"])
    assert lo <= int(f.correct) <= hi, (c, int(f.correct), lo, hi)
    for name, gg, rr in zip(("dh", "dW", "db"), grads, (ref_b["dh"], ref_b["dW"], ref_b["db"])):
        if rr is None:
            assert gg is None, c
            continue
        assert oracle.relative_frobenius(gg, rr) <= TOL_GRAD, (name, c, oracle.relative_frobenius(gg, rr))
    if c["compact"] and nv < c["N"]:
        assert torch.all(grads[0][torch.from_numpy(~valid).cuda()] == 0), c
