"""The oracle against its pins, and each pin set against planted mistakes (CPU only)."""
from __future__ import annotations

import importlib.util
import os
import types

import pytest

import oracle
from tests import oracle_pins as pins

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "flce_oracle.py")


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle)


# Plausible mistakes, each planted in a private copy of the oracle's source: a
# dropped term, a wrong sign or index, a misplaced step of the logit chain.
MUTANTS = {
    "bias dropped": [("x = acc if b is None else acc + widen(b)[None, :]", "x = acc")],
    "bias after scale": [
        ("x = acc if b is None else acc + widen(b)[None, :]", "x = acc"),
        ("x = x * float(logit_scale)",
         "x = x * float(logit_scale) if b is None else x * float(logit_scale) + widen(b)[None, :]")],
    "scale after softcap": [("x = x * float(logit_scale)", "x = x"),
                            ("return c * np.tanh(x / c)", "return c * np.tanh(x / c) * float(logit_scale)")],
    "softcap factor dropped": [("return c * np.tanh(x / c)", "return np.tanh(x / c)")],
    "lse averages": [("return m + np.log(np.exp(z - m[:, None]).sum(axis=1))",
                      "return m + np.log(np.exp(z - m[:, None]).mean(axis=1))")],
    "entropy sign": [("entropy = lse - (p * z).sum(axis=1)", "entropy = lse + (p * z).sum(axis=1)")],
    "argmax ties to highest": [("argmax = z.argmax(axis=1)",
                                "argmax = z.shape[1] - 1 - z[:, ::-1].argmax(axis=1)")],
    "ignored rows in loss": [("loss_tok = np.where(valid, lse - z_t, 0.0)", "loss_tok = lse - z_t")],
    "mean over all tokens": [("denom = float(num_items_in_batch) if num_items_in_batch > 0 else n_valid",
                              "denom = float(num_items_in_batch) if num_items_in_batch > 0 else n_tok")],
    "entropy sum over ignored": [("entropy_sum = float(entropy[valid].sum())",
                                  "entropy_sum = float(entropy.sum())")],
    "grad sign": [("return w[:, None] * (p - onehot) * dz_dacc",
                   "return w[:, None] * (onehot - p) * dz_dacc")],
    "onehot off by one": [("onehot = (t[:, None] == cols[None, :])",
                           "onehot = (t[:, None] == cols[None, :] + 1)")],
    "softcap derivative dropped": [
        ("((1.0 - (z / float(softcap)) ** 2) if softcap > 0.0 else 1.0)", "1.0")],
    "scale derivative dropped": [("dz_dacc = float(logit_scale) * (", "dz_dacc = 1.0 * (")],
    "none ignores upstream grad": [("w = g.copy()", "w = np.ones_like(g)")],
    "mean weight over all tokens": [("g / n_valid if n_valid > 0 else 0.0)", "g / t.shape[0])")],
    "bias grad averaged": [('"db": None if b is None else G.sum(axis=0)',
                            '"db": None if b is None else G.sum(axis=0) / G.shape[0]')],
    "hidden grad transposed head": [('"dh": G @ Wf', '"dh": G @ Wf[::-1]')],
    "num_items ignored in the forward": [("denom = float(num_items_in_batch) if num_items_in_batch > 0 else n_valid",
                                          "denom = n_valid")],
    "num_items ignored in the backward": [("        n_valid = float(num_items_in_batch)", "        pass")],
    "frobenius sqrt dropped": [("den = math.sqrt(float((ref * ref).sum()))", "den = float((ref * ref).sum())"),
                               ("num = math.sqrt(float(((a - ref) ** 2).sum()))",
                                "num = float(((a - ref) ** 2).sum())")],
    "frobenius ratio inverted": [("    return num / den", "    return den / num")],
    "frobenius absolute error": [("    return num / den", "    return num")],
    "frobenius max-abs instead": [("num = math.sqrt(float(((a - ref) ** 2).sum()))",
                                   "num = float(np.abs(a - ref).max()) * math.sqrt(a.size)")],
    "widen through fp32": [('x = x.detach().to("cpu").double().numpy()',
                            'x = x.detach().to("cpu").float().double().numpy()')],
    "widen through bf16": [('x = x.detach().to("cpu").double().numpy()',
                            'x = x.detach().to("cpu").bfloat16().double().numpy()')],
}


def _mutant(edits) -> types.ModuleType:
    src = open(ORACLE_SRC).read()
    for old, new in edits:
        assert src.count(old) >= 1, f"mutation anchor missing: {old!r}"
        src = src.replace(old, new)
    spec = importlib.util.spec_from_loader("flce_oracle_mutant", loader=None)
    mod = importlib.util.module_from_spec(spec)
    exec(compile(src, "flce_oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    mod = _mutant(MUTANTS[name])
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            check(mod)
        except Exception as e:  # an assertion, or the mutant crashing on a shape
            caught.append((check.__name__, type(e).__name__))
    assert caught, f"no pin caught the planted mistake '{name}'"


def test_oracle_matches_frozen_golden():
    """The oracle still reproduces the fixture written by tests/golden/make_golden.py."""
    import json

    import numpy as np

    from tests.golden.make_golden import case
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_small.json")
    gold = json.load(open(path))
    c = case()
    kw = dict(logit_scale=c["logit_scale"], softcap=c["softcap"])
    for red in ("mean", "sum", "none"):
        dl = c["dloss"] if red == "none" else np.array([1.0])
        f = oracle.forward(c["h"], c["W"], c["b"], c["t"], reduction=red, **kw)
        g = oracle.backward(c["h"], c["W"], c["b"], c["t"], reduction=red, dloss=dl, **kw)
        gr = gold[red]
        np.testing.assert_allclose(f["loss"], gr["loss"], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(f["lse"], gr["lse"], rtol=1e-13)
        np.testing.assert_allclose(f["entropy"], gr["entropy"], rtol=1e-13, atol=1e-15)
        assert f["argmax"].tolist() == gr["argmax"]
        assert (f["correct"], f["n_valid"]) == (gr["correct"], gr["n_valid"])
        for k in ("dh", "dW", "db"):
            np.testing.assert_allclose(g[k], gr[k], rtol=1e-12, atol=1e-15)
