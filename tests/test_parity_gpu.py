"""GPU parity of flce_forward / flce_backward (through the C ABI) against the fp64
oracle on the same seeded inputs, at sizes the oracle finishes in seconds that
still span several tiles and ragged tails, plus the edge cases of the method."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from linear_cross_entropy_tmem_gb300.synthetic import TINY, Workload, make_inputs
from tests.parity import TOL_GRAD, TOL_LSE, compare_backward, compare_forward, launch_kinds, run_gpu

pytestmark = pytest.mark.gpu

# name -> (workload, tuning override (chunk columns, dh K splits))
CASES = {
    "tiny N512 D128 V4096 mean": (TINY, (0, 0)),
    "ragged N300 D200 V1000 bias-bf16 s0.7 c5 sum": (
        Workload("r", 300, 200, 1000, sigma_w=0.15, bias=True, logit_scale=0.7, softcap=5.0, reduction="sum",
                 seed=1), (0, 0)),
    "fp32-h N257 D136 V777 bias s0.0625 c30 none": (
        Workload("h32", 257, 136, 777, sigma_w=0.3, hidden_dtype=torch.float32, bias=True, logit_scale=0.0625,
                 softcap=30.0, reduction="none", seed=2), (0, 0)),
    "multi-chunk ksplit3 N384 D256 V3000 bias mean": (
        Workload("mc", 384, 256, 3000, sigma_w=0.1, bias=True, seed=3), (1024, 3)),
    "multi-chunk ksplit1 N640 D512 V2560 none": (
        Workload("mc1", 640, 512, 2560, sigma_w=0.08, reduction="none", seed=4), (768, 1)),
    "fp32-h multi-chunk N200 D64 V1500 softcap sum": (
        Workload("h32mc", 200, 64, 1500, sigma_w=0.4, hidden_dtype=torch.float32, softcap=8.0,
                 reduction="sum", seed=5), (512, 2)),
    "single tile vocab N130 D64 V200 softcap": (
        Workload("v200", 130, 64, 200, sigma_w=0.3, softcap=3.0, seed=6), (0, 0)),
    "minimum D8 V1": (Workload("d8v1", 33, 8, 1, ignore_every=5, seed=7), (0, 0)),
    "D8 V300 mean": (Workload("d8", 70, 8, 300, sigma_w=1.0, seed=8), (0, 0)),
}


@pytest.fixture(autouse=True)
def _reset_tuning():
    from linear_cross_entropy_tmem_gb300.api import testing_set_gemm_mode, testing_set_token_chunk, testing_set_tuning
    yield
    testing_set_tuning(0, 0)
    testing_set_gemm_mode(0)
    testing_set_token_chunk(0)


def _run_case(w: Workload, tuning):
    from linear_cross_entropy_tmem_gb300.api import testing_set_tuning
    testing_set_tuning(*tuning)
    h, W, b, t, dloss = make_inputs(w, "cpu")
    dev = [x.cuda() if x is not None else None for x in (h, W, b, t, dloss)]
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)
    gpu = run_gpu(*dev, **kw)
    assert gpu["status"] == 0
    ref_f = oracle.forward(h, W, b, t, **kw)
    ref_b = oracle.backward(h, W, b, t, dloss=dloss, **kw)
    z = oracle.logits(h, W, b, logit_scale=w.logit_scale, softcap=w.softcap)
    compare_forward(gpu["fwd"], ref_f, reduction=w.reduction, z=z, t=t.numpy())
    compare_backward(gpu["bwd"], ref_b)
    return gpu, dev


@pytest.mark.parametrize("mode", [0, 1, 2], ids=["auto", "single-cta", "cta-pair"])
@pytest.mark.parametrize("name", list(CASES))
def test_parity_small(name, mode):
    from linear_cross_entropy_tmem_gb300.api import testing_set_gemm_mode
    testing_set_gemm_mode(mode)
    w, tuning = CASES[name]
    _run_case(w, tuning)


def test_bitwise_deterministic_across_runs():
    w = CASES["multi-chunk ksplit3 N384 D256 V3000 bias mean"][0]
    from linear_cross_entropy_tmem_gb300.api import testing_set_tuning
    testing_set_tuning(1024, 3)
    h, W, b, t, dloss = [x.cuda() if x is not None else None for x in make_inputs(w, "cpu")]
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)
    a = run_gpu(h, W, b, t, dloss, **kw)
    c = run_gpu(h, W, b, t, dloss, **kw)
    for x, y in zip((a["fwd"].loss, a["fwd"].lse, a["fwd"].entropy, a["fwd"].correct, a["fwd"].entropy_sum),
                    (c["fwd"].loss, c["fwd"].lse, c["fwd"].entropy, c["fwd"].correct, c["fwd"].entropy_sum)):
        assert torch.equal(x, y)
    for x, y in zip(a["bwd"], c["bwd"]):
        assert torch.equal(x, y)


def test_all_ignored_gives_zero_loss_and_exact_zero_grads():
    w = Workload("ign", 100, 64, 500, sigma_w=0.2, bias=True, seed=9)
    for red in ("mean", "sum", "none"):
        h, W, b, t, _ = make_inputs(w, "cuda")
        t[:] = -100
        dloss = torch.ones(100 if red == "none" else 1, device="cuda")
        g = run_gpu(h, W, b, t, dloss, logit_scale=1.0, softcap=0.0, reduction=red)
        f = g["fwd"]
        assert int(f.n_valid) == 0 and int(f.correct) == 0 and float(f.entropy_sum) == 0.0
        assert torch.all(f.loss == 0)
        for x in g["bwd"]:
            assert torch.all(x == 0)


def test_empty_batch():
    import linear_cross_entropy_tmem_gb300 as F
    W = torch.randn(300, 64, device="cuda").to(torch.bfloat16)
    b = torch.randn(300, device="cuda").to(torch.bfloat16)
    h = torch.empty(0, 64, device="cuda", dtype=torch.bfloat16)
    t = torch.empty(0, dtype=torch.int64, device="cuda")
    for red in ("mean", "sum"):
        f = F.flce_forward(h, W, t, b, reduction=red)
        dh, dW, db = F.flce_backward(h, W, t, f.lse, f.n_valid, torch.ones(1, device="cuda"), b, reduction=red)
        torch.cuda.synchronize()
        assert float(f.loss) == 0.0 and int(f.n_valid) == 0 and int(f.correct) == 0
        assert dh.numel() == 0 and torch.all(dW == 0) and torch.all(db == 0)


def test_frozen_head_edge_cases():
    """A frozen head with an empty batch, a one-word vocabulary and an all-ignored batch, through
    every entry point: dhidden is exactly zero and nothing else is written."""
    import linear_cross_entropy_tmem_gb300 as F
    for N, V, ignore_all in ((0, 300, False), (33, 1, False), (700, 3000, True)):
        W = (0.05 * torch.randn(V, 1280, device="cuda")).to(torch.bfloat16)
        b = (0.1 * torch.randn(V, device="cuda")).to(torch.bfloat16)
        h = torch.randn(N, 1280, device="cuda").to(torch.bfloat16)
        t = torch.full((N,), -100, dtype=torch.int64, device="cuda") if ignore_all else \
            torch.randint(0, V, (N,), device="cuda")
        up = torch.ones(1, device="cuda")
        for bwd in ("keep_logits", "recompute"):
            f, (dh, dW, db) = F.flce_forward_backward(h, W, t, up, b, bwd=bwd, frozen_head=True)
            torch.cuda.synchronize()
            assert F.flce_read_device_status(f.workspace) == 0
            assert dW is None and db is None and abs(float(f.loss)) <= 1e-6  # V = 1: lse - z rounds to ~0
            assert dh.shape == h.shape and int(torch.count_nonzero(dh)) == 0
        f = F.flce_forward(h, W, t, b)
        dh, dW, db = F.flce_backward(h, W, t, f.lse, f.n_valid, up, b, frozen_head=True)
        torch.cuda.synchronize()
        assert dW is None and db is None and int(torch.count_nonzero(dh)) == 0


def test_out_of_range_target_sets_status_and_is_ignored():
    w = Workload("oor", 64, 64, 300, sigma_w=0.2, seed=10, ignore_every=0)
    h, W, b, t, dloss = make_inputs(w, "cpu")
    t[5] = 300
    t[9] = -7
    g = run_gpu(h.cuda(), W.cuda(), None, t.cuda(), dloss.cuda(), logit_scale=1.0, softcap=0.0, reduction="mean")
    assert g["status"] == 7
    ref = oracle.forward(h, W, None, t)
    assert ref["status"] == oracle.STATUS_TARGET_OUT_OF_RANGE
    compare_forward(g["fwd"], ref, reduction="mean")
    compare_backward(g["bwd"], oracle.backward(h, W, None, t, dloss=dloss))


def test_targets_at_argmax_give_exact_accuracy():
    """TRL PR #6859, "Correctness": with targets at the argmax, accuracy is exact."""
    for V in (32000, 150000, 200000):
        w = Workload("am", 96, 64, V, sigma_w=0.5, seed=V)
        h, W, b, t, dloss = make_inputs(w, "cpu")
        z = oracle.logits(h, W)
        zs = np.sort(z, axis=1)
        keep = (zs[:, -1] - zs[:, -2]) >= 1e-3          # exclude near-ties
        t = torch.from_numpy(z.argmax(axis=1))
        t[~torch.from_numpy(keep)] = -100
        g = run_gpu(h.cuda(), W.cuda(), None, t.cuda(), dloss.cuda(), logit_scale=1.0, softcap=0.0,
                    reduction="mean", backward=False)
        f = g["fwd"]
        assert int(f.correct) == int(f.n_valid) == int(keep.sum())


def test_ties_go_to_lowest_index():
    """Duplicate head rows give bitwise-equal logits; the lowest index must win.

    Rows 3 and 650 (and 399, 400) are made identical and three times larger than
    the rest, so they hold the maximum for a sizeable share of the tokens.
    """
    w = Workload("tie", 128, 64, 700, sigma_w=0.3, seed=11, ignore_every=0)
    h, W, b, t, dloss = make_inputs(w, "cpu")
    W[3] = (W[3].float() * 3).to(torch.bfloat16)
    W[650] = W[3]
    W[399] = (W[399].float() * 3).to(torch.bfloat16)
    W[400] = W[399]
    z = oracle.logits(h, W)
    am = z.argmax(axis=1)  # first maximum
    zs = np.sort(z, axis=1)
    gap = zs[:, -1] - zs[:, -2]
    exact = np.isin(am, [3, 399])
    assert exact.sum() >= 10 and np.all(gap[exact] == 0.0)
    t = torch.from_numpy(am)
    g = run_gpu(h.cuda(), W.cuda(), None, t.cuda(), dloss.cuda(), logit_scale=1.0, softcap=0.0,
                reduction="sum", backward=False)
    may_flip = int(((gap > 0) & (gap < 1e-3)).sum())
    assert 128 - may_flip <= int(g["fwd"].correct) <= 128


def test_autograd_wrapper_matches_direct_calls():
    import linear_cross_entropy_tmem_gb300 as F
    w = CASES["ragged N300 D200 V1000 bias-bf16 s0.7 c5 sum"][0]
    h, W, b, t, _ = [x.cuda() if x is not None else None for x in make_inputs(w, "cpu")]
    hh, WW, bb = (x.clone().requires_grad_(True) for x in (h, W, b))
    loss, correct, n_valid, ent = F.linear_cross_entropy(hh, WW, t, bb, logit_scale=0.7, softcap=5.0,
                                                         reduction="sum")
    (2.0 * loss).backward()
    f = F.flce_forward(h, W, t, b, logit_scale=0.7, softcap=5.0, reduction="sum")
    dh, dW, db = F.flce_backward(h, W, t, f.lse, f.n_valid, torch.full((1,), 2.0, device="cuda"), b,
                                 logit_scale=0.7, softcap=5.0, reduction="sum")
    torch.cuda.synchronize()
    assert torch.equal(loss, f.loss)
    assert torch.equal(hh.grad, dh) and torch.equal(WW.grad, dW) and torch.equal(bb.grad, db)


def test_scale_gradient_is_one_fp32_multiply_and_rounding():
    """flce_scale_gradient: x = rn(x * s) in place, bit for bit what an fp32 multiply followed by one
    rounding to the buffer's dtype gives; s == 1 leaves the buffer untouched."""
    import linear_cross_entropy_tmem_gb300 as F
    g = torch.Generator().manual_seed(31)
    for dt in (torch.bfloat16, torch.float32):
        x0 = (torch.randn(100003, generator=g) * 3).to(dt).cuda()
        for s in (2.5, -0.37, 1.0, 0.0):
            x = x0.clone()
            F.scale_gradient(x, torch.full((1,), s, device="cuda"))
            torch.cuda.synchronize()
            assert torch.equal(x, (x0.float() * s).to(dt)), (dt, s)


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("D", [200, 1280], ids=["recompute", "keep-logits"])
def test_autograd_gradients_in_forward(D, reduction):
    """The autograd wrapper computes mean / sum gradients in the forward (fused call with an upstream
    gradient of 1) and scales them by the upstream gradient in the backward; 'none' keeps the
    separate backward.  Checked against the oracle with a non-power-of-two upstream gradient, and a
    second backward through the same graph (retain_graph) accumulates the same gradient again."""
    import linear_cross_entropy_tmem_gb300 as F
    w = Workload("ag", 700, D, 3000, sigma_w=0.1, bias=True, softcap=10.0, reduction=reduction, seed=15)
    hc, Wc, bc, tc, dc = make_inputs(w, "cpu")
    h, W, b, t = (x.cuda() for x in (hc, Wc, bc, tc))
    up = dc.cuda() if reduction == "none" else torch.full((), 2.5, device="cuda")
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=reduction)
    ref_b = oracle.backward(hc, Wc, bc, tc, dloss=up.cpu().reshape(-1), **kw)
    hh, WW, bb = (x.clone().requires_grad_(True) for x in (h, W, b))
    loss, correct, n_valid, ent = F.linear_cross_entropy(hh, WW, t, bb, **kw)
    loss.backward(up, retain_graph=True)
    torch.cuda.synchronize()
    compare_backward((hh.grad, WW.grad, bb.grad), ref_b)
    first = [x.grad.clone() for x in (hh, WW, bb)]
    loss.backward(up)  # recomputed: the saved gradients were scaled in place by the first backward
    torch.cuda.synchronize()
    for x, g1 in zip((hh, WW, bb), first):
        assert oracle.relative_frobenius(x.grad.float().cpu(), 2 * g1.float().cpu()) <= 1e-2
    hh2, WW2, bb2 = (x.clone().requires_grad_(True) for x in (h, W, b))
    loss2, *_ = F.linear_cross_entropy(hh2, WW2, t, bb2, grad_in_forward=False, **kw)
    assert torch.equal(loss, loss2)
    loss2.backward(up)
    torch.cuda.synchronize()
    for g1, x in zip(first, (hh2, WW2, bb2)):
        assert oracle.relative_frobenius(g1.float().cpu(), x.grad.float().cpu()) <= 1e-2


@pytest.mark.parametrize("D", [200, 1280], ids=["recompute", "keep-logits"])
def test_autograd_none_backward_through_slices(D):
    """Reduction 'none' through the autograd wrapper: backpropagating loss[:k].sum() (retain_graph)
    and then loss[k:].sum() gives the gradient of loss.sum() (Liger-Kernel PR #1574, review reply
    point 2: backward through slices of the per-token losses keeps working).  Each dhidden row
    depends on its own token's upstream weight only, so it is the same bits as a single backward;
    dweight and dbias add two rounded partial sums, so they match to rounding and the oracle."""
    import linear_cross_entropy_tmem_gb300 as F
    w = Workload("slices", 700, D, 3000, sigma_w=0.1, bias=True, softcap=10.0, reduction="none", seed=17)
    hc, Wc, bc, tc, _ = make_inputs(w, "cpu")
    h, W, b, t = (x.cuda() for x in (hc, Wc, bc, tc))
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction="none")
    k = 700 // 3
    hh, WW, bb = (x.clone().requires_grad_(True) for x in (h, W, b))
    loss, *_ = F.linear_cross_entropy(hh, WW, t, bb, **kw)
    loss[:k].sum().backward(retain_graph=True)
    loss[k:].sum().backward()
    h1, W1, b1 = (x.clone().requires_grad_(True) for x in (h, W, b))
    loss1, *_ = F.linear_cross_entropy(h1, W1, t, b1, **kw)
    loss1.sum().backward()
    torch.cuda.synchronize()
    assert torch.equal(hh.grad, h1.grad)
    for a, c in ((WW.grad, W1.grad), (bb.grad, b1.grad)):
        assert oracle.relative_frobenius(a.float().cpu(), c.float().cpu()) <= 5e-3
    ref_b = oracle.backward(hc, Wc, bc, tc, dloss=torch.ones(700), **kw)
    compare_backward((hh.grad, WW.grad, bb.grad), ref_b)


# ---------------------------------------------------------------------------
# num_items_in_batch and valid-token compaction
# ---------------------------------------------------------------------------
def test_num_items_in_batch_matches_oracle():
    """TRL PR #6859 review, "Test coverage" item 10: the mean over a caller-given count."""
    w = CASES["ragged N300 D200 V1000 bias-bf16 s0.7 c5 sum"][0].scaled(reduction="mean")
    h, W, b, t, dloss = make_inputs(w, "cpu")
    dloss = torch.full((1,), 0.7)
    dev = [x.cuda() if x is not None else None for x in (h, W, b, t, dloss)]
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction="mean")
    for items in (1000.0, 37.0):
        g = run_gpu(*dev, num_items_in_batch=items, **kw)
        ref_f = oracle.forward(h, W, b, t, num_items_in_batch=items, **kw)
        ref_b = oracle.backward(h, W, b, t, dloss=dloss, num_items_in_batch=items, **kw)
        compare_forward(g["fwd"], ref_f, reduction="mean")
        compare_backward(g["bwd"], ref_b)


def _compare_compacted(gpu, ref_f, ref_b, t, reduction):
    valid = ref_f["valid"]
    f = gpu["fwd"]
    lse = f.lse.double().cpu().numpy()
    ent = f.entropy.double().cpu().numpy()
    np.testing.assert_allclose(lse[valid], ref_f["lse"][valid], atol=2e-3, rtol=0)
    np.testing.assert_allclose(ent[valid], ref_f["entropy"][valid], atol=5e-3, rtol=0)
    assert np.all(lse[~valid] == 0.0) and np.all(ent[~valid] == 0.0)
    nv = int(f.n_valid)
    assert nv == ref_f["n_valid"]
    if reduction == "none":
        np.testing.assert_allclose(f.loss.double().cpu().numpy(), ref_f["loss"], atol=2e-3, rtol=0)
    else:
        tol = 2e-3 * (nv if reduction == "sum" else 1)
        assert abs(float(f.loss) - ref_f["loss"]) <= tol
    assert abs(float(f.entropy_sum) - ref_f["entropy_sum"]) <= 5e-3 * max(1, nv)
    assert int(f.correct) == ref_f["correct"]
    dh, dW, db = gpu["bwd"]
    assert torch.all(dh[torch.from_numpy(~valid).cuda()] == 0)
    assert oracle.relative_frobenius(dh, ref_b["dh"]) <= 1e-2
    assert oracle.relative_frobenius(dW, ref_b["dW"]) <= 1e-2
    if db is not None:
        assert oracle.relative_frobenius(db, ref_b["db"]) <= 1e-2


COMPACT_CASES = ["tiny N512 D128 V4096 mean", "ragged N300 D200 V1000 bias-bf16 s0.7 c5 sum",
                 "fp32-h N257 D136 V777 bias s0.0625 c30 none", "multi-chunk ksplit3 N384 D256 V3000 bias mean",
                 "multi-chunk ksplit1 N640 D512 V2560 none", "fp32-h multi-chunk N200 D64 V1500 softcap sum"]


@pytest.mark.parametrize("mode", [0, 1, 2], ids=["auto", "single-cta", "cta-pair"])
@pytest.mark.parametrize("name", COMPACT_CASES)
@pytest.mark.parametrize("ignore_every", [17, 3])
def test_compaction_matches_oracle(name, mode, ignore_every):
    """FLCE_FLAG_COMPACT_VALID: valid tokens match the oracle; ignored ones get 0."""
    from linear_cross_entropy_tmem_gb300.api import testing_set_gemm_mode, testing_set_tuning
    w, tuning = CASES[name]
    w = w.scaled(ignore_every=ignore_every)
    testing_set_gemm_mode(mode)
    testing_set_tuning(*tuning)
    h, W, b, t, dloss = make_inputs(w, "cpu")
    dev = [x.cuda() if x is not None else None for x in (h, W, b, t, dloss)]
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)
    gpu = run_gpu(*dev, compact=True, **kw)
    assert gpu["status"] == 0
    _compare_compacted(gpu, oracle.forward(h, W, b, t, **kw), oracle.backward(h, W, b, t, dloss=dloss, **kw),
                       t, w.reduction)


def test_compaction_all_ignored_and_out_of_range():
    w = Workload("cign", 300, 64, 700, sigma_w=0.2, bias=True, seed=12)
    h, W, b, t, _ = make_inputs(w, "cuda")
    t[:] = -100
    g = run_gpu(h, W, b, t, torch.ones(1, device="cuda"), logit_scale=1.0, softcap=0.0, reduction="mean",
                compact=True)
    assert int(g["fwd"].n_valid) == 0 and float(g["fwd"].loss) == 0.0
    for x in g["bwd"]:
        assert torch.all(x == 0)
    t[:] = 5
    t[7] = 700  # out of range: reported and treated as ignored
    g = run_gpu(h, W, b, t, torch.ones(1, device="cuda"), logit_scale=1.0, softcap=0.0, reduction="mean",
                compact=True)
    assert g["status"] == 7 and int(g["fwd"].n_valid) == 299


def test_compaction_is_deterministic():
    from linear_cross_entropy_tmem_gb300.api import testing_set_tuning
    w, tuning = CASES["multi-chunk ksplit3 N384 D256 V3000 bias mean"]
    testing_set_tuning(*tuning)
    h, W, b, t, dloss = [x.cuda() if x is not None else None for x in make_inputs(w.scaled(ignore_every=3), "cpu")]
    a = run_gpu(h, W, b, t, dloss, logit_scale=1.0, softcap=0.0, reduction="mean", compact=True)
    c = run_gpu(h, W, b, t, dloss, logit_scale=1.0, softcap=0.0, reduction="mean", compact=True)
    assert torch.equal(a["fwd"].lse, c["fwd"].lse) and torch.equal(a["fwd"].loss, c["fwd"].loss)
    for x, y in zip(a["bwd"], c["bwd"]):
        assert torch.equal(x, y)


# ---------------------------------------------------------------------------
# flce_forward_backward: one call, same results as forward then backward
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("mode", [0, 1, 2], ids=["auto", "single-cta", "cta-pair"])
@pytest.mark.parametrize("compact", [False, True], ids=["all-tokens", "compact"])
@pytest.mark.parametrize("name", ["ragged N300 D200 V1000 bias-bf16 s0.7 c5 sum",
                                  "fp32-h N257 D136 V777 bias s0.0625 c30 none",
                                  "multi-chunk ksplit3 N384 D256 V3000 bias mean"])
def test_fused_call_equals_separate_calls(name, compact, mode):
    import linear_cross_entropy_tmem_gb300 as F
    from linear_cross_entropy_tmem_gb300.api import testing_set_gemm_mode, testing_set_tuning
    w, tuning = CASES[name]
    testing_set_gemm_mode(mode)
    testing_set_tuning(*tuning)
    h, W, b, t, dloss = [x.cuda() if x is not None else None for x in make_inputs(w, "cpu")]
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction, compact=compact,
              num_items_in_batch=500.0 if w.reduction == "mean" else 0.0)
    sep = run_gpu(h, W, b, t, dloss, **kw)
    fwd, grads = F.flce_forward_backward(h, W, t, dloss, b, entropy=True, bwd="recompute", **kw)
    torch.cuda.synchronize()
    assert F.flce_read_device_status(fwd.workspace) == 0
    for x, y in ((fwd.loss, sep["fwd"].loss), (fwd.lse, sep["fwd"].lse), (fwd.entropy, sep["fwd"].entropy),
                 (fwd.correct, sep["fwd"].correct), (fwd.n_valid, sep["fwd"].n_valid),
                 (fwd.entropy_sum, sep["fwd"].entropy_sum)):
        assert torch.equal(x, y)
    for x, y in zip(grads, sep["bwd"]):
        assert (x is None and y is None) or torch.equal(x, y)
    if not compact:
        ref_f = oracle.forward(h.cpu(), W.cpu(), None if b is None else b.cpu(), t.cpu(),
                               logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction,
                               num_items_in_batch=kw["num_items_in_batch"])
        compare_forward(fwd, ref_f, reduction=w.reduction)


# ---------------------------------------------------------------------------
# Token-chunked backward of the fused call (kept fp32 logits, 6NVD)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [256, 0], ids=["chunk256", "auto-chunk"])
@pytest.mark.parametrize("mode", [0, 1, 2], ids=["auto", "single-cta", "cta-pair"])
@pytest.mark.parametrize("name", list(CASES))
def test_keep_logits_parity(name, mode, chunk):
    """Every output of the token-chunked fused call against the oracle, element by element, with
    several token chunks (ragged last chunk) and the dh K split of the case; a batch of at most 256
    tokens is one chunk (dW and dbias written straight from it)."""
    import linear_cross_entropy_tmem_gb300 as F
    from linear_cross_entropy_tmem_gb300.api import testing_set_gemm_mode, testing_set_token_chunk, testing_set_tuning
    w, tuning = CASES[name]
    testing_set_gemm_mode(mode)
    testing_set_tuning(*tuning)
    testing_set_token_chunk(chunk)
    hc, Wc, bc, tc, dc = make_inputs(w, "cpu")
    h, W, b, t, dloss = [x.cuda() if x is not None else None for x in (hc, Wc, bc, tc, dc)]
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)
    (fwd, grads), kinds = launch_kinds(
        lambda: F.flce_forward_backward(h, W, t, dloss, b, entropy=True, bwd="keep_logits", **kw))
    assert F.flce_read_device_status(fwd.workspace) == 0
    chunks = kinds.count("bwd_logit_grad")
    assert (chunks == 1 if w.n_tokens <= 256 else chunks >= 2) and "bwd_recompute" not in kinds
    assert kinds.count("fwd_logits") == kinds.count("bwd_dhidden") == kinds.count("bwd_dweight") == chunks
    ref_f = oracle.forward(hc, Wc, bc, tc, **kw)
    ref_b = oracle.backward(hc, Wc, bc, tc, dloss=dc, **kw)
    z = oracle.logits(hc, Wc, bc, logit_scale=w.logit_scale, softcap=w.softcap)
    compare_forward(fwd, ref_f, reduction=w.reduction, z=z, t=tc.numpy())
    compare_backward(grads, ref_b)


@pytest.mark.parametrize("mode", [0, 1, 2], ids=["auto", "single-cta", "cta-pair"])
@pytest.mark.parametrize("ignore_every", [17, 3])
@pytest.mark.parametrize("name", list(COMPACT_CASES))
def test_keep_logits_with_compaction(name, ignore_every, mode):
    """Kept logits over the compacted tokens: 256-row chunks of the valid tokens (a partial chunk
    and, with a third of the tokens ignored, chunks with no valid row at all), or one chunk for a
    batch of at most 256 tokens."""
    import linear_cross_entropy_tmem_gb300 as F
    from linear_cross_entropy_tmem_gb300.api import testing_set_gemm_mode, testing_set_token_chunk, testing_set_tuning
    w, tuning = CASES[name]
    w = w.scaled(ignore_every=ignore_every)
    testing_set_gemm_mode(mode)
    testing_set_tuning(*tuning)
    testing_set_token_chunk(256)
    h, W, b, t, dloss = make_inputs(w, "cpu")
    dev = [x.cuda() if x is not None else None for x in (h, W, b, t, dloss)]
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)
    (fwd, grads), kinds = launch_kinds(lambda: F.flce_forward_backward(
        dev[0], dev[1], dev[3], dev[4], dev[2], entropy=True, compact=True, bwd="keep_logits", **kw))
    assert F.flce_read_device_status(fwd.workspace) == 0
    chunks = kinds.count("bwd_logit_grad")
    assert (chunks == 1 if w.n_tokens <= 256 else chunks >= 2) and "bwd_recompute" not in kinds
    _compare_compacted({"fwd": fwd, "bwd": grads}, oracle.forward(h, W, b, t, **kw),
                       oracle.backward(h, W, b, t, dloss=dloss, **kw), t, w.reduction)


@pytest.mark.parametrize("n_tokens", [700, 200], ids=["chunks", "one-chunk"])
@pytest.mark.parametrize("compact", [False, True], ids=["all-tokens", "compact"])
@pytest.mark.parametrize("reduction,items", [("mean", 0.0), ("mean", 700.0), ("sum", 0.0), ("none", 0.0)])
def test_keep_logits_reductions_and_all_ignored(reduction, items, compact, n_tokens):
    """The mean's denominator (counted before the first chunk, or num_items_in_batch), the other
    reductions, and an all-ignored batch (zero loss, exact zero gradients) on the token path, with
    several 256-token chunks and with a batch of at most 256 tokens as one chunk."""
    import linear_cross_entropy_tmem_gb300 as F
    from linear_cross_entropy_tmem_gb300.api import testing_set_token_chunk
    testing_set_token_chunk(256)
    w = Workload("kl", n_tokens, 256, 3000, sigma_w=0.1, bias=True, reduction=reduction, ignore_every=5, seed=11)
    hc, Wc, bc, tc, dc = make_inputs(w, "cpu")
    for targets in (tc, torch.full_like(tc, -100)):
        h, W, b, t, dloss = [x.cuda() for x in (hc, Wc, bc, targets, dc)]
        kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=reduction, num_items_in_batch=items)
        fwd, grads = F.flce_forward_backward(h, W, t, dloss, b, entropy=True, bwd="keep_logits", compact=compact,
                                             **kw)
        torch.cuda.synchronize()
        assert F.flce_read_device_status(fwd.workspace) == 0
        ref_f = oracle.forward(hc, Wc, bc, targets, **kw)
        ref_b = oracle.backward(hc, Wc, bc, targets, dloss=dc, **kw)
        if compact:  # compaction writes lse = entropy = 0 at ignored tokens: compare the valid ones
            v = torch.from_numpy(ref_f["valid"]).cuda()
            fwd = fwd._replace(lse=torch.where(v, fwd.lse, 0.0), entropy=torch.where(v, fwd.entropy, 0.0))
            ref_f = dict(ref_f, lse=np.where(ref_f["valid"], ref_f["lse"], 0.0),
                         entropy=np.where(ref_f["valid"], ref_f["entropy"], 0.0))
            assert torch.all(fwd.lse[~v] == 0)
        compare_forward(fwd, ref_f, reduction=reduction)
        if int(ref_f["n_valid"]) == 0:
            assert all(int(torch.count_nonzero(g)) == 0 for g in grads)
        else:
            compare_backward(grads, ref_b)


def test_keep_logits_is_deterministic():
    import linear_cross_entropy_tmem_gb300 as F
    from linear_cross_entropy_tmem_gb300.api import testing_set_token_chunk
    testing_set_token_chunk(256)
    w, _ = CASES["multi-chunk ksplit1 N640 D512 V2560 none"]
    h, W, b, t, dloss = [x.cuda() if x is not None else None for x in make_inputs(w, "cpu")]
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction, bwd="keep_logits")
    a = F.flce_forward_backward(h, W, t, dloss, b, entropy=True, **kw)
    c = F.flce_forward_backward(h, W, t, dloss, b, entropy=True, **kw)
    for x, y in zip((a[0].loss, a[0].lse, a[0].entropy, *a[1][:2]), (c[0].loss, c[0].lse, c[0].entropy, *c[1][:2])):
        assert torch.equal(x, y)


# ---------------------------------------------------------------------------
# Guard regions: no kernel writes past the end of an output or the workspace
# ---------------------------------------------------------------------------
CANARY = 0x5A


def _guarded(n_bytes):
    """A device byte buffer with 4 KB of canary after the first n_bytes."""
    return torch.full((n_bytes + 4096,), CANARY, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("mode", [1, 2], ids=["single-cta", "cta-pair"])
@pytest.mark.parametrize("compact", [False, True], ids=["all-tokens", "compact"])
@pytest.mark.parametrize("name", ["ragged N300 D200 V1000 bias-bf16 s0.7 c5 sum",
                                  "fp32-h N257 D136 V777 bias s0.0625 c30 none",
                                  "multi-chunk ksplit3 N384 D256 V3000 bias mean"])
def test_no_writes_past_outputs_or_workspace(name, compact, mode):
    import ctypes

    import linear_cross_entropy_tmem_gb300.api as api
    from linear_cross_entropy_tmem_gb300 import binding as B
    from linear_cross_entropy_tmem_gb300.api import testing_set_gemm_mode, testing_set_tuning
    w, tuning = CASES[name]
    testing_set_gemm_mode(mode)
    testing_set_tuning(*tuning)
    h, W, b, t, dloss = [x.cuda() if x is not None else None for x in make_inputs(w, "cpu")]
    N, D, V = w.n_tokens, w.hidden, w.vocab
    prob = api.make_problem(N, D, V, hidden_dtype=h.dtype, bias_dtype=b.dtype if b is not None else torch.bfloat16,
                            logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction, compact=compact)
    f32, hb = 4, h.element_size()
    sizes = {"loss": (N if w.reduction == "none" else 1) * f32, "lse": N * f32, "ent": N * f32, "corr": 8, "nv": 8,
             "es": f32, "ws_f": api.flce_workspace_size(prob, 0), "ws_b": api.flce_workspace_size(prob, 1),
             "dh": N * D * hb, "dW": V * D * 2, "db": V * b.element_size() if b is not None else 0}
    bufs = {k: _guarded(v) for k, v in sizes.items()}
    p = {k: ctypes.c_void_p(v.data_ptr()) for k, v in bufs.items()}
    ptr = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())  # noqa: E731
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    lib = B.load()
    B.check(lib.flce_forward(ctypes.byref(prob), ptr(h), ptr(W), ptr(b), ptr(t), p["loss"], p["lse"], p["ent"],
                             p["corr"], p["nv"], p["es"], p["ws_f"], sizes["ws_f"], s), "forward")
    B.check(lib.flce_backward(ctypes.byref(prob), ptr(h), ptr(W), ptr(b), ptr(t), p["lse"], p["nv"], ptr(dloss),
                              p["dh"], p["dW"], p["db"] if b is not None else None, p["ws_b"], sizes["ws_b"], s),
            "backward")
    torch.cuda.synchronize()
    for k, buf in bufs.items():
        tail = buf[sizes[k]:]
        assert torch.all(tail == CANARY), f"write past the end of {k}"
    # the guarded buffers hold the results the parity tests check
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)
    hc, Wc, bc, tc, dc = [x.cpu() if x is not None else None for x in (h, W, b, t, dloss)]
    ref_f = oracle.forward(hc, Wc, bc, tc, **kw)
    ref_b = oracle.backward(hc, Wc, bc, tc, dloss=dc, **kw)
    assert int(bufs["nv"][:8].view(torch.int64).item()) == ref_f["n_valid"]
    lse = bufs["lse"][:sizes["lse"]].view(torch.float32).cpu().double().numpy()
    valid = ref_f["valid"]
    assert np.abs(lse[valid] - ref_f["lse"][valid]).max() <= TOL_LSE
    if compact:  # compaction leaves ignored rows out of the matmul and writes lse 0 for them
        assert np.all(lse[~valid] == 0.0)
    dh = bufs["dh"][:sizes["dh"]].view(h.dtype).view(N, D)
    dW = bufs["dW"][:sizes["dW"]].view(torch.bfloat16).view(V, D)
    db = None if b is None else bufs["db"][:sizes["db"]].view(b.dtype)
    compare_backward((dh, dW, db), ref_b)


@pytest.mark.parametrize("mode", [1, 2], ids=["single-cta", "cta-pair"])
@pytest.mark.parametrize("name", ["ragged N300 D200 V1000 bias-bf16 s0.7 c5 sum",
                                  "fp32-h N257 D136 V777 bias s0.0625 c30 none",
                                  "multi-chunk ksplit3 N384 D256 V3000 bias mean",
                                  "single tile vocab N130 D64 V200 softcap", "D8 V300 mean"])
def test_keep_logits_no_writes_past_outputs_or_workspace(name, mode):
    """Canary tails after every output and the workspace of the token-chunked fused call."""
    import ctypes

    import linear_cross_entropy_tmem_gb300.api as api
    from linear_cross_entropy_tmem_gb300 import binding as B
    from linear_cross_entropy_tmem_gb300.api import testing_set_gemm_mode, testing_set_token_chunk, testing_set_tuning
    w, tuning = CASES[name]
    testing_set_gemm_mode(mode)
    testing_set_tuning(*tuning)
    testing_set_token_chunk(256)
    hc, Wc, bc, tc, dc = make_inputs(w, "cpu")
    h, W, b, t, dloss = [x.cuda() if x is not None else None for x in (hc, Wc, bc, tc, dc)]
    N, D, V = w.n_tokens, w.hidden, w.vocab
    prob = api.make_problem(N, D, V, hidden_dtype=h.dtype, bias_dtype=b.dtype if b is not None else torch.bfloat16,
                            logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction, bwd="keep_logits")
    f32, hb = 4, h.element_size()
    sizes = {"loss": (N if w.reduction == "none" else 1) * f32, "lse": N * f32, "ent": N * f32, "corr": 8, "nv": 8,
             "es": f32, "ws": api.flce_workspace_size(prob, 2), "dh": N * D * hb, "dW": V * D * 2,
             "db": V * b.element_size() if b is not None else 0}
    bufs = {k: _guarded(v) for k, v in sizes.items()}
    p = {k: ctypes.c_void_p(v.data_ptr()) for k, v in bufs.items()}
    ptr = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())  # noqa: E731
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    B.check(B.load().flce_forward_backward(ctypes.byref(prob), ptr(h), ptr(W), ptr(b), ptr(t), ptr(dloss), p["loss"],
                                           p["lse"], p["ent"], p["corr"], p["nv"], p["es"], p["dh"], p["dW"],
                                           p["db"] if b is not None else None, p["ws"], sizes["ws"], s),
            "forward_backward")
    torch.cuda.synchronize()
    for k, buf in bufs.items():
        assert torch.all(buf[sizes[k]:] == CANARY), f"write past the end of {k}"
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)
    ref_b = oracle.backward(hc, Wc, bc, tc, dloss=dc, **kw)
    dh = bufs["dh"][:sizes["dh"]].view(h.dtype).view(N, D)
    dW = bufs["dW"][:sizes["dW"]].view(torch.bfloat16).view(V, D)
    db = None if b is None else bufs["db"][:sizes["db"]].view(b.dtype)
    compare_backward((dh, dW, db), ref_b)


# ---------------------------------------------------------------------------
# fp32 operands: an fp32 head (with fp32 hidden states); two- and three-term splits
# ---------------------------------------------------------------------------
def _fp32_head(W_bf16: torch.Tensor, seed: int) -> torch.Tensor:
    """An fp32 head close to the bf16 one whose values use all 24 significand bits."""
    g = torch.Generator().manual_seed(seed)
    return (W_bf16.float() * (1.0 + 0.01 * torch.randn(W_bf16.shape, generator=g))).contiguous()


FP32_CASES = {
    "fp32-h N257 D136 V777 bias s0.0625 c30 none": CASES["fp32-h N257 D136 V777 bias s0.0625 c30 none"][0],
    "fp32-h multi-chunk N200 D64 V1500 softcap sum": CASES["fp32-h multi-chunk N200 D64 V1500 softcap sum"][0],
    "fp32-h N700 D256 V3000 bias mean": Workload("h32w32", 700, 256, 3000, sigma_w=0.1, hidden_dtype=torch.float32,
                                                 bias=True, seed=13),
}


@pytest.mark.parametrize("full", [False, True], ids=["two-term", "three-term"])
@pytest.mark.parametrize("entry", ["separate", "fused-recompute", "fused-keep", "fused-keep-compact"])
@pytest.mark.parametrize("name", list(FP32_CASES))
def test_fp32_head_parity(name, entry, full):
    """fp32 hidden states with an fp32 head (FLCE_F32 weight, fp32 dweight) on every entry point."""
    import linear_cross_entropy_tmem_gb300 as F
    from linear_cross_entropy_tmem_gb300.api import testing_set_token_chunk
    testing_set_token_chunk(256)
    w = FP32_CASES[name]
    h, Wb, b, t, dloss = make_inputs(w, "cpu")
    W = _fp32_head(Wb, w.seed)
    dev = [x.cuda() if x is not None else None for x in (h, W, b, t, dloss)]
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)
    ref_f = oracle.forward(h, W, b, t, **kw)
    ref_b = oracle.backward(h, W, b, t, dloss=dloss, **kw)
    if entry == "separate":
        gpu = run_gpu(*dev, fp32_full=full, **kw)
        assert gpu["status"] == 0
        fwd, grads = gpu["fwd"], gpu["bwd"]
    else:
        bwd = "recompute" if entry == "fused-recompute" else "keep_logits"
        fwd, grads = F.flce_forward_backward(dev[0], dev[1], dev[3], dev[4], dev[2], entropy=True, bwd=bwd,
                                             compact=entry.endswith("compact"), fp32_full=full, **kw)
        torch.cuda.synchronize()
        assert F.flce_read_device_status(fwd.workspace) == 0
    assert grads[1].dtype == torch.float32
    if entry.endswith("compact"):
        _compare_compacted({"fwd": fwd, "bwd": grads}, ref_f, ref_b, t, w.reduction)
        return
    z = oracle.logits(h, W, b, logit_scale=w.logit_scale, softcap=w.softcap)
    compare_forward(fwd, ref_f, reduction=w.reduction, z=z, t=t.numpy())
    compare_backward(grads, ref_b)


@pytest.mark.parametrize("fp32_head", [False, True], ids=["bf16-head", "fp32-head"])
def test_fp32_full_removes_operand_rounding(fp32_head):
    """Three-term splits carry all 24 bits of fp32 operands.  With one MMA step (K = 16) the
    operands' rounding dominates the two-term error, and the three-term lse error against the exact
    fp64 logits drops to the level of fp32 arithmetic.  At K = 512 the tensor core's fp32
    accumulation (about K/16 ulps of the accumulator) dominates both, so the split must only not
    make it worse."""
    import linear_cross_entropy_tmem_gb300 as F
    for D, check in ((16, "operand"), (512, "accumulation")):
        N, V = 512, 4096
        g = torch.Generator().manual_seed(21 + D)
        h = torch.randn(N, D, generator=g)                    # fp32 with all 24 bits used
        W = torch.randn(V, D, generator=g) * (10.0 / D ** 0.5)  # logits of order 10
        if not fp32_head:
            W = W.to(torch.bfloat16)
        t = torch.randint(0, V, (N,), generator=g)
        ref = oracle.forward(h, W, None, t)
        err = {}
        for full in (False, True):
            f = F.flce_forward(h.cuda(), W.cuda(), t.cuda(), None, fp32_full=full)
            torch.cuda.synchronize()
            err[full] = float(np.abs(f.lse.double().cpu().numpy() - ref["lse"]).max())
        if check == "operand":
            # each of the (3 or 6) term products is one accumulation step of at most ~1 ulp of the
            # accumulator (|logit| <= ~48 here, ulp 3.8e-6), plus the lse's own fp32 arithmetic
            nseg = 6 if fp32_head else 3
            assert err[True] <= (nseg + 4) * 3.8e-6, (D, err)
            assert 4 * err[True] <= err[False], (D, err)
        else:
            assert err[True] <= 1.2 * err[False] and err[True] <= 5e-4, (D, err)


@pytest.mark.parametrize("entry", ["fused-keep", "fused-recompute", "separate"])
def test_cuda_graph_capture_replays_bitwise(entry):
    """The entry points enqueue only kernels and async memsets on the caller's stream, with no host
    synchronisation and no allocation, so a step can be captured into a CUDA graph once and replayed;
    each replay gives the eager results bit for bit (after one eager call, which also does the
    library's one-time per-device set-up)."""
    import linear_cross_entropy_tmem_gb300 as F
    import linear_cross_entropy_tmem_gb300.api as api
    from linear_cross_entropy_tmem_gb300.api import testing_set_token_chunk
    testing_set_token_chunk(256)
    w = Workload("graph", 700, 256, 3000, sigma_w=0.1, bias=True, softcap=20.0, reduction="mean", seed=16)
    h, W, b, t, dloss = [x.cuda() for x in make_inputs(w, "cpu")]
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction)
    bwd = {"fused-keep": "keep_logits", "fused-recompute": "recompute", "separate": "auto"}[entry]
    prob = api.make_problem(700, 256, 3000, bias_dtype=b.dtype, bwd=bwd, **kw)
    f32 = dict(dtype=torch.float32, device="cuda")
    outs = dict(loss=torch.empty(1, **f32), lse=torch.empty(700, **f32), ent=torch.empty(700, **f32),
                corr=torch.empty(1, dtype=torch.int64, device="cuda"), nv=torch.empty(1, dtype=torch.int64, device="cuda"),
                es=torch.empty(1, **f32), dh=torch.empty_like(h), dW=torch.empty_like(W), db=torch.empty_like(b))
    if entry == "separate":
        ws_f = torch.empty(api.flce_workspace_size(prob, 0), dtype=torch.uint8, device="cuda")
        ws_b = torch.empty(api.flce_workspace_size(prob, 1), dtype=torch.uint8, device="cuda")
    else:
        ws = torch.empty(api.flce_workspace_size(prob, 2), dtype=torch.uint8, device="cuda")
    import ctypes

    from linear_cross_entropy_tmem_gb300 import binding as B
    lib = B.load()
    ptr = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731

    def step():
        s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        o = outs
        if entry == "separate":
            B.check(lib.flce_forward(ctypes.byref(prob), ptr(h), ptr(W), ptr(b), ptr(t), ptr(o["loss"]), ptr(o["lse"]),
                                     ptr(o["ent"]), ptr(o["corr"]), ptr(o["nv"]), ptr(o["es"]), ptr(ws_f),
                                     ws_f.numel(), s), "forward")
            B.check(lib.flce_backward(ctypes.byref(prob), ptr(h), ptr(W), ptr(b), ptr(t), ptr(o["lse"]), ptr(o["nv"]),
                                      ptr(dloss), ptr(o["dh"]), ptr(o["dW"]), ptr(o["db"]), ptr(ws_b), ws_b.numel(), s),
                    "backward")
        else:
            B.check(lib.flce_forward_backward(ctypes.byref(prob), ptr(h), ptr(W), ptr(b), ptr(t), ptr(dloss),
                                              ptr(o["loss"]), ptr(o["lse"]), ptr(o["ent"]), ptr(o["corr"]),
                                              ptr(o["nv"]), ptr(o["es"]), ptr(o["dh"]), ptr(o["dW"]), ptr(o["db"]),
                                              ptr(ws), ws.numel(), s), "forward_backward")

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # eager: the reference results, and the library's one-time set-up
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in outs.items()}
    for v in outs.values():
        v.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        for v in outs.values():
            v.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for k in ref:
            assert torch.equal(outs[k], ref[k]), k
    ref_f = oracle.forward(h.cpu(), W.cpu(), b.cpu(), t.cpu(), **kw)
    assert abs(float(outs["loss"]) - ref_f["loss"]) <= 2e-3


@pytest.mark.parametrize("entry", ["fused-keep", "fused-recompute", "separate"])
@pytest.mark.parametrize("variant", ["bias-softcap", "fp32h-compact"])
def test_frozen_head_forms_dhidden_only(entry, variant):
    """FLCE_FLAG_FROZEN_HEAD (a head that is not trained, as in LoRA): no dweight / dbias product is
    launched and none is written; the forward outputs and dhidden are the same bits as with the head
    trained, and dhidden matches the oracle.  Kept logits in 256-token chunks with a ragged last one."""
    import linear_cross_entropy_tmem_gb300 as F
    from linear_cross_entropy_tmem_gb300.api import testing_set_token_chunk
    testing_set_token_chunk(256)
    if variant == "bias-softcap":
        w = Workload("fz1", 700, 1280, 3000, sigma_w=0.05, bias=True, softcap=20.0, reduction="mean", seed=51)
        compact = False
    else:
        w = Workload("fz2", 600, 1280, 2600, sigma_w=0.05, hidden_dtype=torch.float32, bias=True,
                     logit_scale=0.5, reduction="none", ignore_every=3, seed=52)
        compact = True
    hc, Wc, bc, tc, dc = make_inputs(w, "cpu")
    h, W, b, t, dloss = [x.cuda() for x in (hc, Wc, bc, tc, dc)]
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction, compact=compact)

    def run(frozen):
        if entry == "separate":
            f = F.flce_forward(h, W, t, b, entropy=True, **kw)
            return f, F.flce_backward(h, W, t, f.lse, f.n_valid, dloss, b, frozen_head=frozen, **kw)
        bwd = "keep_logits" if entry == "fused-keep" else "recompute"
        return F.flce_forward_backward(h, W, t, dloss, b, entropy=True, bwd=bwd, frozen_head=frozen, **kw)

    (ff, gf), kinds = launch_kinds(lambda: run(True))
    assert "bwd_dweight" not in kinds and "bwd_dhidden" in kinds
    assert gf[1] is None and gf[2] is None
    fa, ga = run(False)
    torch.cuda.synchronize()
    for x, y in zip((ff.loss, ff.lse, ff.entropy, ff.correct, ff.n_valid, ff.entropy_sum, gf[0]),
                    (fa.loss, fa.lse, fa.entropy, fa.correct, fa.n_valid, fa.entropy_sum, ga[0])):
        assert torch.equal(x, y)
    ref_b = oracle.backward(hc, Wc, bc, tc, dloss=dc, **{k: v for k, v in kw.items() if k != "compact"})
    assert oracle.relative_frobenius(gf[0], ref_b["dh"]) <= TOL_GRAD


def test_autograd_frozen_head():
    """The autograd wrapper forms dhidden only when neither the weight nor the bias requires a
    gradient: the hidden gradient is the same bits as with the head trained."""
    import linear_cross_entropy_tmem_gb300 as F
    w = Workload("fz3", 700, 1280, 3000, sigma_w=0.05, bias=True, softcap=10.0, reduction="mean", seed=53)
    h, W, b, t, _ = [x.cuda() for x in make_inputs(w, "cpu")]
    kw = dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction="mean")
    h1 = h.clone().requires_grad_(True)
    loss1, *_ = F.linear_cross_entropy(h1, W, t, b, **kw)  # W and b do not require gradients
    loss1.backward(torch.full((), 1.5, device="cuda"))
    h2, W2, b2 = h.clone().requires_grad_(True), W.clone().requires_grad_(True), b.clone().requires_grad_(True)
    loss2, *_ = F.linear_cross_entropy(h2, W2, t, b2, **kw)
    loss2.backward(torch.full((), 1.5, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(loss1, loss2) and torch.equal(h1.grad, h2.grad)
    assert W.grad is None and b.grad is None


def test_two_host_threads_at_once():
    """Two host threads call the library at once, each on its own stream with its own problem (one
    kept-logits, one recompute): every result is the same bits as the same call made alone."""
    import threading

    import linear_cross_entropy_tmem_gb300 as F
    ws_ = [Workload("th1", 900, 1280, 3000, sigma_w=0.05, bias=True, softcap=15.0, seed=61),
           Workload("th2", 500, 512, 5000, sigma_w=0.05, reduction="sum", seed=62)]
    inputs = [[x.cuda() if x is not None else None for x in make_inputs(w, "cpu")] for w in ws_]

    def call(i):
        h, W, b, t, dloss = inputs[i]
        w = ws_[i]
        f, g = F.flce_forward_backward(h, W, t, dloss, b, entropy=True, logit_scale=w.logit_scale,
                                       softcap=w.softcap, reduction=w.reduction)
        return [f.loss, f.lse, f.entropy, f.correct, f.n_valid, f.entropy_sum, *[x for x in g if x is not None]]

    alone = []
    for i in range(2):
        alone.append([x.clone() for x in call(i)])
        torch.cuda.synchronize()
    out, errors = [None, None], []

    def worker(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                res = [call(i) for _ in range(3)]
            s.synchronize()
            out[i] = res
        except Exception as e:  # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for i in range(2):
        for res in out[i]:
            for x, y in zip(res, alone[i]):
                assert torch.equal(x, y), i


def test_back_to_back_calls_on_one_stream():
    """The GEMMs are launched as programmatic dependents (they set up while the kernel before them
    finishes, and wait for its results before touching global memory).  Calls of different shapes
    and algorithms enqueued back to back on one stream, with no synchronisation between them, give
    the same bits as each call run alone; the second call of a shape reuses the first one's
    workspace."""
    import linear_cross_entropy_tmem_gb300 as F
    from linear_cross_entropy_tmem_gb300.api import testing_set_token_chunk
    testing_set_token_chunk(256)
    cases = [
        (Workload("b2b1", 1100, 2304, 4000, sigma_w=0.02, bias=True, softcap=30.0, reduction="mean", seed=31),
         dict(bwd="keep_logits")),
        (Workload("b2b2", 300, 256, 3000, sigma_w=0.1, reduction="none", seed=32), dict(bwd="recompute")),
        (Workload("b2b3", 700, 1280, 2600, sigma_w=0.05, hidden_dtype=torch.float32, bias=True, logit_scale=0.5,
                  reduction="sum", ignore_every=3, seed=33), dict(bwd="auto", compact=True)),
    ]
    inputs = [[x.cuda() if x is not None else None for x in make_inputs(w, "cpu")] for w, _ in cases]
    kws = [dict(logit_scale=w.logit_scale, softcap=w.softcap, reduction=w.reduction, **extra) for w, extra in cases]

    def call(i, ws=None):
        h, W, b, t, dloss = inputs[i]
        return F.flce_forward_backward(h, W, t, dloss, b, entropy=True, workspace=ws, **kws[i])

    def flat(res):
        f, g = res
        return [f.loss, f.lse, f.entropy, f.correct, f.n_valid, f.entropy_sum, *[x for x in g if x is not None]]

    alone = []
    for i in range(len(cases)):
        alone.append([x.clone() for x in flat(call(i))])
        torch.cuda.synchronize()
    order = [0, 1, 2, 0, 2, 1]
    results = []
    first = {}
    for i in order:  # no synchronisation in between
        res = call(i, first[i].workspace if i in first else None)
        first.setdefault(i, res[0])
        results.append((i, res))
    torch.cuda.synchronize()
    for i, res in results:
        assert F.flce_read_device_status(res[0].workspace) == 0
        for x, y in zip(flat(res), alone[i]):
            assert torch.equal(x, y), i


@pytest.mark.parametrize("softcap", [0.0, 30.0], ids=["plain", "softcap"])
def test_nan_hidden_row_stays_in_its_row(softcap):
    """A NaN in one hidden row makes every logit of that row NaN, so its loss, lse and dh row are
    NaN (no clamp or maximum may turn it into a finite value), while every other row keeps the
    oracle's values: rows are independent until dW and the reductions sum over them."""
    import linear_cross_entropy_tmem_gb300 as F
    w = Workload("nan", 300, 200, 1000, sigma_w=0.15, softcap=softcap, reduction="none", seed=21)
    h, W, b, t, dloss = make_inputs(w, "cpu")
    bad = int(np.flatnonzero(t.numpy() != -100)[20])  # a valid token
    h_nan = h.clone()
    h_nan[bad, 5] = float("nan")
    kw = dict(softcap=softcap, reduction="none")
    f = F.flce_forward(h_nan.cuda(), W.cuda(), t.cuda(), entropy=True, **kw)
    g = F.flce_backward(h_nan.cuda(), W.cuda(), t.cuda(), f.lse, f.n_valid, dloss.cuda(), **kw)
    torch.cuda.synchronize()
    assert F.flce_read_device_status(f.workspace) == 0
    ref = oracle.forward(h, W, None, t, **kw)
    ref_b = oracle.backward(h, W, None, t, dloss=dloss, **kw)
    keep = np.arange(w.n_tokens) != bad
    lse, loss, dh = f.lse.cpu().numpy(), f.loss.cpu().numpy(), g[0].float().cpu().numpy()
    assert np.isnan(lse[bad]) and np.isnan(dh[bad]).all()
    assert np.isnan(loss[bad])
    assert np.abs(lse[keep] - ref["lse"][keep]).max() < TOL_LSE
    assert np.abs(loss[keep] - ref["loss_tok"][keep]).max() < TOL_LSE
    ref_dh = ref_b["dh"][keep]
    assert np.linalg.norm(dh[keep] - ref_dh) <= 1e-2 * np.linalg.norm(ref_dh)


@pytest.mark.parametrize("where", ["hidden", "weight", "dhidden", "dweight", "workspace"])
@pytest.mark.parametrize("host", ["pinned", "pageable"])
def test_host_pointers_are_refused_before_any_launch(where, host):
    """The tensor maps and the products address this GPU's memory only: a host pointer (pinned or
    pageable) for an operand, a gradient or the workspace is refused with FLCE_ERR_INVALID_ARG before
    anything is enqueued, so the outputs keep their fill and the status word is untouched."""
    import ctypes

    import linear_cross_entropy_tmem_gb300.api as api
    from linear_cross_entropy_tmem_gb300 import binding as B
    lib = B.load()
    w = Workload("host-ptr", 300, 64, 1000, sigma_w=0.2, seed=41)
    h, W, _, t, dloss = (x.cuda() if x is not None else None for x in make_inputs(w, "cpu"))
    prob = api.make_problem(300, 64, 1000)
    f32 = dict(dtype=torch.float32, device="cuda")
    loss = torch.full((1,), float("nan"), **f32)
    lse = torch.full((300,), float("nan"), **f32)
    correct = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    n_valid = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    ent = torch.full((1,), float("nan"), **f32)
    dh = torch.full_like(h, float("nan"))
    dW = torch.full_like(W, float("nan"))
    ws = torch.full((api.flce_workspace_size(prob, 2),), 0x5A, dtype=torch.uint8, device="cuda")
    args = {"hidden": h, "weight": W, "dhidden": dh, "dweight": dW, "workspace": ws}
    src = args[where]
    raw = torch.empty(src.numel() * src.element_size() + 256, dtype=torch.uint8,
                      pin_memory=(host == "pinned"))
    off = (-raw.data_ptr()) % 256  # 256-byte aligned like the device buffers, so only the location differs
    args[where] = raw[off:off + src.numel() * src.element_size()].view(src.dtype).view(src.shape)
    args[where].copy_(src.cpu())
    p = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())  # noqa: E731
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.flce_forward_backward(ctypes.byref(prob), p(args["hidden"]), p(args["weight"]), None, p(t), p(dloss),
                                   p(loss), p(lse), None, p(correct), p(n_valid), p(ent), p(args["dhidden"]),
                                   p(args["dweight"]), None, p(args["workspace"]), args["workspace"].numel(), s)
    assert rc == B.FLCE_ERR_INVALID_ARG
    if where in ("hidden", "weight", "workspace"):
        rws = torch.full((api.flce_workspace_size(prob, 0),), 0x5A, dtype=torch.uint8, device="cuda")
        if where == "workspace":
            rws = args["workspace"]
        rc = lib.flce_forward(ctypes.byref(prob), p(args["hidden"]), p(args["weight"]), None, p(t), p(loss),
                              p(lse), None, p(correct), p(n_valid), p(ent), p(rws), rws.numel(), s)
        assert rc == B.FLCE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.isnan(loss).all() and torch.isnan(lse).all() and int(correct) == -1 and int(n_valid) == -1
    assert torch.isnan(dh).all() and torch.isnan(dW).all()
    if where != "workspace":
        assert bool((ws == 0x5A).all())
