"""Checks that pin the fp64 oracle to things other than itself.

Each ``check_*`` takes an oracle namespace ``o`` (the real ``oracle`` package or
a copy with a planted mistake) and raises ``AssertionError`` when the oracle
disagrees with what the pages or the mathematics fix:

* library routines it must reduce to in special cases
  (``torch.nn.functional.cross_entropy``, ``scipy.stats.entropy``);
* closed forms (zero head, saturated soft cap, one-word vocabulary);
* invariants (entropy in [0, log V], gradient rows summing to zero, ...);
* central finite differences of its own forward (pins the backward);
* brute force with Python's ``math`` module and an exact-arithmetic
  evaluation with sympy on tiny inputs;
* TRL PR #6859 "Correctness": with targets set to the argmax, accuracy is exact
  at V = 32000, 150000 and 200000.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import torch
import torch.nn.functional as F

IGN = -100


def _rand_case(seed, n=7, d=5, v=11, bias=False, ignore=(2,), scale=1.0):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((n, d))
    W = rng.standard_normal((v, d)) * 0.7
    b = rng.standard_normal(v) * 0.3 if bias else None
    t = rng.integers(0, v, n)
    for i in ignore:
        if i < n:
            t[i] = IGN
    return h, W, b, t


def _torch_logits(h, W, b, scale):
    z = torch.from_numpy(h) @ torch.from_numpy(W).T
    if b is not None:
        z = z + torch.from_numpy(b)[None, :]
    return z * scale


def check_forward_matches_torch(o):
    """No soft cap: the loss is torch's cross_entropy on ``s * (h W^T + b)`` (fp64)."""
    for seed, bias, scale in [(0, False, 1.0), (1, True, 1.0), (2, True, 0.37), (3, False, 2.5)]:
        h, W, b, t = _rand_case(seed, bias=bias, ignore=(1, 4))
        z = _torch_logits(h, W, b, scale)
        tt = torch.from_numpy(t)
        for red in ("mean", "sum", "none"):
            out = o.forward(h, W, b, t, logit_scale=scale, reduction=red)
            ref = F.cross_entropy(z, tt, ignore_index=IGN, reduction=red).numpy()
            np.testing.assert_allclose(out["loss"], ref, rtol=1e-12, atol=1e-12)
        out = o.forward(h, W, b, t, logit_scale=scale)
        np.testing.assert_allclose(out["lse"], torch.logsumexp(z, dim=1).numpy(), rtol=1e-13)
        assert np.array_equal(out["argmax"], torch.argmax(z, dim=1).numpy())
        assert out["n_valid"] == int((tt != IGN).sum())


def check_entropy_matches_scipy(o):
    """Per-token entropy equals ``-sum p log p`` of the softmax (scipy.stats.entropy)."""
    from scipy.special import softmax
    from scipy.stats import entropy
    for seed, cap in [(4, 0.0), (5, 3.0)]:
        h, W, b, t = _rand_case(seed, bias=True)
        out = o.forward(h, W, b, t, logit_scale=0.8, softcap=cap)
        x = (h @ W.T + b) * 0.8
        z = cap * np.tanh(x / cap) if cap > 0 else x
        ref = entropy(softmax(z, axis=1), axis=1)
        np.testing.assert_allclose(out["entropy"], ref, rtol=1e-11, atol=1e-12)
        valid = t != IGN
        np.testing.assert_allclose(out["entropy_sum"], ref[valid].sum(), rtol=1e-11)


def check_softcap_limits(o):
    """Soft cap: ``c -> inf`` recovers the uncapped loss; saturation gives a closed form."""
    h, W, b, t = _rand_case(6, bias=True)
    a = o.forward(h, W, b, t, logit_scale=0.5, softcap=0.0)
    big = o.forward(h, W, b, t, logit_scale=0.5, softcap=1e7)
    np.testing.assert_allclose(big["loss"], a["loss"], rtol=1e-9)
    # Saturation: one hidden unit, logits +-1000 before the cap.  With c = 2 and
    # s = 0.5 every z is exactly +-2 in fp64, so lse = log(k e^2 + (V-k) e^-2).
    v = 9
    signs = np.array([1, -1, -1, 1, -1, -1, -1, 1, -1], dtype=np.float64)
    W1 = (signs * 2000.0)[:, None]
    h1 = np.ones((3, 1))
    t1 = np.array([0, 1, IGN])
    out = o.forward(h1, W1, None, t1, logit_scale=0.5, softcap=2.0, reduction="none")
    k = int((signs > 0).sum())
    lse = math.log(k * math.exp(2.0) + (v - k) * math.exp(-2.0))
    np.testing.assert_allclose(out["lse"], lse, rtol=1e-14)
    np.testing.assert_allclose(out["loss"], [lse - 2.0, lse + 2.0, 0.0], rtol=1e-14, atol=1e-15)
    # c bounds |z|: the per-token loss never exceeds log V + 2c.
    assert np.all(out["loss_tok"] <= math.log(v) + 4.0 + 1e-12)


def _scalar_loss(o, h, W, b, t, red, dloss, **kw):
    out = o.forward(h, W, b, t, reduction=red, **kw)
    if red == "none":
        return float(np.dot(out["loss"], dloss))
    return float(out["loss"]) * float(dloss[0])


def check_gradients_finite_difference(o):
    """Central differences of the forward pin dh, dW and db (all reductions, cap, bias)."""
    eps = 1e-6
    for red, cap, bias, scale in itertools.product(("mean", "sum", "none"), (0.0, 2.5),
                                                   (False, True), (1.0, 0.7)):
        h, W, b, t = _rand_case(7, n=4, d=3, v=5, bias=bias, ignore=(2,))
        rng = np.random.default_rng(8)
        dloss = rng.uniform(0, 2, 4) if red == "none" else np.array([1.3])
        kw = dict(logit_scale=scale, softcap=cap)
        g = o.backward(h, W, b, t, reduction=red, dloss=dloss, **kw)
        for name, arr in (("dh", h), ("dW", W), ("db", b)):
            if arr is None:
                assert g["db"] is None
                continue
            num = np.zeros_like(arr)
            for idx in np.ndindex(arr.shape):
                old = arr[idx]
                arr[idx] = old + eps
                lp = _scalar_loss(o, h, W, b, t, red, dloss, **kw)
                arr[idx] = old - eps
                lm = _scalar_loss(o, h, W, b, t, red, dloss, **kw)
                arr[idx] = old
                num[idx] = (lp - lm) / (2 * eps)
            np.testing.assert_allclose(g[name], num, rtol=1e-6, atol=1e-8,
                                       err_msg=f"{name} red={red} cap={cap} bias={bias} s={scale}")


def check_zero_head_closed_form(o):
    """W = 0, b = 0: z = 0, so lse = H = log V, argmax 0, dh = 0 and dW, db in closed form."""
    rng = np.random.default_rng(9)
    n, d, v, s = 6, 4, 7, 0.6
    h = rng.standard_normal((n, d))
    W = np.zeros((v, d))
    b = np.zeros(v)
    t = np.array([0, 3, IGN, 0, 6, 2])
    valid = t != IGN
    for red in ("mean", "sum", "none"):
        dloss = rng.uniform(0, 2, n) if red == "none" else np.array([0.9])
        out = o.forward(h, W, b, t, logit_scale=s, reduction=red)
        np.testing.assert_allclose(out["lse"], math.log(v), rtol=1e-15)
        np.testing.assert_allclose(out["entropy"], math.log(v), rtol=1e-14)
        assert np.all(out["argmax"] == 0)
        assert out["correct"] == int(((t == 0) & valid).sum())
        exp_loss = {"mean": math.log(v), "sum": valid.sum() * math.log(v)}
        if red == "none":
            np.testing.assert_allclose(out["loss"], np.where(valid, math.log(v), 0.0), rtol=1e-15)
        else:
            np.testing.assert_allclose(out["loss"], exp_loss[red], rtol=1e-14)
        g = o.backward(h, W, b, t, logit_scale=s, reduction=red, dloss=dloss)
        assert np.all(g["dh"] == 0.0)
        if red == "none":
            w = np.where(valid, dloss, 0.0)
        elif red == "sum":
            w = np.where(valid, dloss[0], 0.0)
        else:
            w = np.where(valid, dloss[0] / valid.sum(), 0.0)
        dW = np.zeros((v, d))
        db = np.zeros(v)
        for i in range(n):
            for j in range(v):
                coef = s * w[i] * (1.0 / v - (1.0 if t[i] == j else 0.0))
                dW[j] += coef * h[i]
                db[j] += coef
        np.testing.assert_allclose(g["dW"], dW, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(g["db"], db, rtol=1e-13, atol=1e-15)


def check_invariants(o):
    """0 <= H <= log V, loss >= 0, lse >= max z, gradient rows sum to 0, sum_v db = 0."""
    for seed in (10, 11, 12):
        h, W, b, t = _rand_case(seed, n=9, d=6, v=13, bias=True, ignore=(0, 5))
        for cap in (0.0, 1.5):
            out = o.forward(h, W, b, t, logit_scale=1.3, softcap=cap, reduction="none")
            z = o.logits(h, W, b, logit_scale=1.3, softcap=cap)
            assert np.all(out["entropy"] >= -1e-12) and np.all(out["entropy"] <= math.log(13) + 1e-12)
            assert np.all(out["loss"] >= 0.0)
            assert np.all(out["lse"] >= z.max(axis=1))
            assert np.all(out["loss"][t == IGN] == 0.0)
        # no soft cap: each gradient row sums to zero, so the bias gradient sums to zero
        G = o.grad_logits(h, W, b, t, logit_scale=1.3, reduction="sum", dloss=np.array([1.0]))
        np.testing.assert_allclose(G.sum(axis=1), 0.0, atol=1e-14)
        g = o.backward(h, W, b, t, logit_scale=1.3, reduction="sum", dloss=np.array([1.0]))
        np.testing.assert_allclose(g["db"].sum(), 0.0, atol=1e-13)
        # all rows of W equal: logits equal along the vocabulary, so dh = 0
        Wc = np.tile(W[:1], (13, 1))
        g = o.backward(h, Wc, None, t, reduction="mean", dloss=np.array([1.0]))
        np.testing.assert_allclose(g["dh"], 0.0, atol=1e-15)


def check_all_ignored(o):
    """Every target ignored: loss 0, exactly zero gradients (TRL PR #6859 review, item 5)."""
    h, W, b, _ = _rand_case(13, bias=True)
    t = np.full(h.shape[0], IGN)
    for red in ("mean", "sum", "none"):
        dloss = np.ones(h.shape[0]) if red == "none" else np.array([1.0])
        out = o.forward(h, W, b, t, reduction=red, softcap=2.0)
        assert out["n_valid"] == 0 and out["correct"] == 0 and out["entropy_sum"] == 0.0
        assert np.all(np.asarray(out["loss"]) == 0.0)
        g = o.backward(h, W, b, t, reduction=red, dloss=dloss, softcap=2.0)
        for k in ("dh", "dW", "db"):
            assert np.all(g[k] == 0.0), k


def check_vocab_one(o):
    """V = 1: the only class has probability 1, so loss 0 and entropy 0."""
    h, W, b, _ = _rand_case(14, v=1, bias=True, ignore=())
    t = np.zeros(h.shape[0], dtype=np.int64)
    out = o.forward(h, W, b, t, reduction="none", softcap=3.0, logit_scale=0.5)
    np.testing.assert_allclose(out["loss"], 0.0, atol=1e-15)
    np.testing.assert_allclose(out["entropy"], 0.0, atol=1e-15)
    assert out["correct"] == h.shape[0]


def check_argmax_targets_exact_accuracy(o):
    """TRL PR #6859, "Correctness": targets = argmax give exact accuracy at V = 32000, 150000, 200000."""
    for v in (32000, 150000, 200000):
        rng = np.random.default_rng(v)
        h = rng.standard_normal((5, 8))
        W = rng.standard_normal((v, 8)) * 0.02
        z = h @ W.T
        t = z.argmax(axis=1)
        t[3] = IGN
        out = o.forward(h, W, None, t)
        assert out["correct"] == out["n_valid"] == 4
        t2 = (t + 1) % v
        t2[3] = IGN
        assert o.forward(h, W, None, t2)["correct"] == 0


def check_ties_lowest_index(o):
    """Equal largest logits: the argmax is the lowest index (torch / NumPy convention)."""
    W = np.array([[0.0], [2.0], [1.0], [2.0], [2.0]])
    h = np.array([[1.0], [1.0]])
    out = o.forward(h, W, None, np.array([1, 3]), reduction="none")
    assert list(out["argmax"]) == [1, 1]
    assert out["correct"] == 1


def check_brute_force_python(o):
    """Tiny case by explicit loops over Python floats (math.fsum), soft cap and bias on."""
    h, W, b, t = _rand_case(15, n=3, d=2, v=4, bias=True, ignore=(1,))
    s, c = 0.9, 1.7
    out = o.forward(h, W, b, t, logit_scale=s, softcap=c, reduction="none")
    for i in range(3):
        zs = []
        for j in range(4):
            acc = math.fsum(float(h[i, k]) * float(W[j, k]) for k in range(2))
            zs.append(c * math.tanh((acc + float(b[j])) * s / c))
        lse = math.log(math.fsum(math.exp(zj) for zj in zs))
        ps = [math.exp(zj - lse) for zj in zs]
        ent = -math.fsum(pj * math.log(pj) for pj in ps)
        assert abs(out["lse"][i] - lse) < 1e-14
        assert abs(out["entropy"][i] - ent) < 1e-14
        exp_loss = 0.0 if t[i] == IGN else lse - zs[t[i]]
        assert abs(out["loss"][i] - exp_loss) < 1e-14


def check_sympy_exact(o):
    """A rational-input case evaluated with sympy at 40 digits (independent arithmetic)."""
    import sympy as sp
    hq = [[sp.Rational(1, 2), sp.Rational(-3, 4)], [sp.Rational(5, 8), sp.Rational(1, 8)]]
    Wq = [[sp.Rational(1, 4), sp.Rational(1, 2)], [sp.Rational(-1, 2), sp.Rational(3, 8)],
          [sp.Rational(7, 8), sp.Rational(-1, 4)]]
    bq = [sp.Rational(1, 16), sp.Rational(-1, 8), sp.Rational(0)]
    s, c = sp.Rational(3, 4), sp.Rational(5, 2)
    t = [2, 0]
    h = np.array([[float(x) for x in r] for r in hq])
    W = np.array([[float(x) for x in r] for r in Wq])
    b = np.array([float(x) for x in bq])
    out = o.forward(h, W, b, np.array(t), logit_scale=0.75, softcap=2.5, reduction="none")
    for i in range(2):
        z = [c * sp.tanh((sum(hq[i][k] * Wq[j][k] for k in range(2)) + bq[j]) * s / c) for j in range(3)]
        lse = sp.log(sum(sp.exp(zj) for zj in z))
        loss = sp.N(lse - z[t[i]], 40)
        ent = sp.N(lse - sum(sp.exp(zj - lse) * zj for zj in z), 40)
        assert abs(out["loss"][i] - float(loss)) < 1e-14
        assert abs(out["entropy"][i] - float(ent)) < 1e-14


def check_subset_helpers(o):
    """Row/column subset helpers equal the whole-matrix results."""
    h, W, b, t = _rand_case(16, n=10, d=4, v=9, bias=True, ignore=(3,))
    rng = np.random.default_rng(17)
    dloss = rng.uniform(0, 2, 10)
    kw = dict(logit_scale=0.8, softcap=2.0)
    for red in ("mean", "sum", "none"):
        dl = dloss if red == "none" else np.array([1.1])
        full_f = o.forward(h, W, b, t, reduction=red, **kw)
        full_b = o.backward(h, W, b, t, reduction=red, dloss=dl, **kw)
        rows = np.array([0, 3, 7, 9])
        sub = o.forward_rows(h, W, b, t, rows, **kw)
        np.testing.assert_allclose(sub["lse"], full_f["lse"][rows], rtol=1e-14)
        np.testing.assert_allclose(o.lse_all(h, W, b, row_block=3, **kw), full_f["lse"], rtol=1e-14)
        dh = o.dhidden_rows(h, W, b, t, rows, n_valid=full_f["n_valid"], reduction=red, dloss=dl, **kw)
        np.testing.assert_allclose(dh, full_b["dh"][rows], rtol=1e-12, atol=1e-15)
        vr = np.array([1, 4, 8])
        dW, db = o.dweight_rows(h, W, b, t, vr, full_f["lse"], reduction=red, dloss=dl, **kw)
        np.testing.assert_allclose(dW, full_b["dW"][vr], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(db, full_b["db"][vr], rtol=1e-12, atol=1e-15)


def check_out_of_range_target(o):
    """A target outside [0, V) that is not the ignore index is reported and treated as ignored."""
    h, W, b, t = _rand_case(18, ignore=())
    t2 = t.copy()
    t2[2] = W.shape[0] + 3
    out = o.forward(h, W, b, t2, reduction="none")
    assert out["status"] == o.STATUS_TARGET_OUT_OF_RANGE
    assert out["loss"][2] == 0.0 and out["n_valid"] == h.shape[0] - 1
    assert o.forward(h, W, b, t, reduction="none")["status"] == o.STATUS_OK


def check_num_items_in_batch(o):
    """The mean over num_items_in_batch equals the summed loss divided by it; its
    gradient is pinned by central differences of that forward."""
    h, W, b, t = _rand_case(19, n=4, d=3, v=5, bias=True, ignore=(1,))
    kw = dict(logit_scale=0.8, softcap=2.0)
    total = o.forward(h, W, b, t, reduction="sum", **kw)["loss"]
    for items in (3.0, 7.0, 64.0):
        m = o.forward(h, W, b, t, reduction="mean", num_items_in_batch=items, **kw)["loss"]
        assert abs(m - total / items) <= 1e-15 * max(1.0, abs(total))
        g = o.backward(h, W, b, t, reduction="mean", dloss=np.array([1.5]), num_items_in_batch=items, **kw)
        eps = 1e-6
        for name, arr in (("dh", h), ("dW", W), ("db", b)):
            num = np.zeros_like(arr)
            for idx in np.ndindex(arr.shape):
                old = arr[idx]
                arr[idx] = old + eps
                lp = o.forward(h, W, b, t, reduction="mean", num_items_in_batch=items, **kw)["loss"]
                arr[idx] = old - eps
                lm = o.forward(h, W, b, t, reduction="mean", num_items_in_batch=items, **kw)["loss"]
                arr[idx] = old
                num[idx] = 1.5 * (lp - lm) / (2 * eps)
            np.testing.assert_allclose(g[name], num, rtol=1e-6, atol=1e-9, err_msg=f"{name} items={items}")
    # 0 means "use n_valid"
    a = o.forward(h, W, b, t, reduction="mean", num_items_in_batch=0.0, **kw)["loss"]
    assert abs(a - total / 3) <= 1e-15 * max(1.0, abs(total))


def check_rows_independent(o):
    """Tokens are independent until the sums over them: a NaN in one hidden row makes exactly that
    row's lse, loss and dh row NaN and leaves every other row's lse, loss, entropy and dh as they
    were (the GPU NaN test compares the other rows with the oracle on the clean input)."""
    h, W, b, t = _rand_case(91, n=6, d=5, v=13, bias=True)
    dl = np.linspace(0.5, 1.5, 6)
    keep = np.arange(6) != 3
    assert t[3] != IGN
    for softcap in (0.0, 4.0):
        kw = dict(logit_scale=0.8, softcap=softcap, reduction="none")
        ref_f = o.forward(h, W, b, t, **kw)
        ref_b = o.backward(h, W, b, t, dloss=dl, **kw)
        hn = h.copy()
        hn[3, 1] = np.nan
        f = o.forward(hn, W, b, t, **kw)
        g = o.backward(hn, W, b, t, dloss=dl, **kw)
        assert np.isnan(f["lse"][3]) and np.isnan(f["loss_tok"][3]) and np.isnan(g["dh"][3]).all()
        for key in ("lse", "loss_tok", "entropy"):
            np.testing.assert_allclose(f[key][keep], ref_f[key][keep], rtol=1e-13, atol=0)
        np.testing.assert_allclose(g["dh"][keep], ref_b["dh"][keep], rtol=1e-12, atol=1e-300)


def check_relative_frobenius(o):
    """The gradient tolerance's measure against values worked out by hand: ``||a - ref||_F /
    ||ref||_F`` with a difference (3, 4) (norm 5) over a reference (6, 8) (norm 10) is exactly 0.5;
    it is scale-invariant (a relative, not an absolute, error), not symmetric in its arguments, 0 for
    two zero arrays and infinite for a nonzero array against a zero reference.  It widens bf16, fp32
    and fp64 torch tensors as well as NumPy arrays."""
    ref = np.array([[0.0, 0.0], [6.0, 8.0]])
    a = ref + np.array([[3.0, 4.0], [0.0, 0.0]])
    assert o.relative_frobenius(a, ref) == 0.5
    assert o.relative_frobenius(ref, a) == 5.0 / math.sqrt(9.0 + 16.0 + 36.0 + 64.0)
    for k in (1e-3, 3.7, -2.0, 1e6):
        assert abs(o.relative_frobenius(k * a, k * ref) - 0.5) < 1e-15
    assert o.relative_frobenius(np.zeros((2, 3)), np.zeros((2, 3))) == 0.0
    assert o.relative_frobenius(np.ones(3), np.zeros(3)) == math.inf
    # every entry here is a small integer, exact in bf16 and fp32
    for dt in (torch.bfloat16, torch.float32, torch.float64):
        assert o.relative_frobenius(torch.tensor(a, dtype=dt), torch.tensor(ref, dtype=dt)) == 0.5
    # one entry off by 1 in a 4 x 4 reference of twos: sqrt(1) / sqrt(16 * 4) = 1/8
    r = np.full((4, 4), 2.0)
    x = r.copy()
    x[1, 2] = 3.0
    assert o.relative_frobenius(torch.tensor(x, dtype=torch.bfloat16), r) == 0.125


def check_widen_exact(o):
    """Widening is exact: bf16 1/3 is 0.333984375 (8 significant bits, rounded to nearest), fp32
    1/3 is 11184811 / 2^25, and an fp64 tensor keeps every bit; bf16 / fp32 NumPy-side inputs
    widen to the same values."""
    third = torch.tensor([1.0 / 3.0], dtype=torch.float64)
    assert o.widen(third.to(torch.bfloat16))[0] == 0.333984375
    assert o.widen(third.to(torch.float32))[0] == 11184811.0 / 2.0 ** 25
    assert o.widen(third)[0] == 1.0 / 3.0
    assert o.widen(np.float32(1.0 / 3.0)) == 11184811.0 / 2.0 ** 25
    tiny = torch.tensor([2.0 ** -133, -(2.0 ** 100) * 1.5], dtype=torch.float64)
    assert o.widen(tiny.to(torch.bfloat16)).tolist() == [2.0 ** -133, -(2.0 ** 100) * 1.5]
    assert o.widen(tiny.to(torch.float32)).dtype == np.float64


ALL_CHECKS = [
    check_forward_matches_torch, check_entropy_matches_scipy, check_softcap_limits,
    check_gradients_finite_difference, check_zero_head_closed_form, check_invariants,
    check_all_ignored, check_vocab_one, check_argmax_targets_exact_accuracy,
    check_ties_lowest_index, check_brute_force_python, check_sympy_exact,
    check_subset_helpers, check_out_of_range_target, check_num_items_in_batch, check_rows_independent,
    check_relative_frobenius, check_widen_exact,
]
