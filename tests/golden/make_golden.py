"""Writes ``oracle_small.json``: a hand-listed tiny case and the oracle's outputs for it.

The pages print no worked example that can be reproduced without trained
weights, so this fixture only freezes the oracle's own answer on a small,
exactly representable input (every value is a multiple of 1/16, exact in
bf16).  It guards the oracle against silent changes; the oracle itself is
pinned by the checks in ``tests/oracle_pins.py``.  Calls only ``oracle/``.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def case():
    n, d, v = 4, 8, 6
    h = np.array([[((i * 7 + k * 3) % 11 - 5) / 16.0 for k in range(d)] for i in range(n)])
    W = np.array([[((j * 5 + k * 2) % 13 - 6) / 16.0 for k in range(d)] for j in range(v)])
    b = np.array([(j % 3 - 1) / 16.0 for j in range(v)])
    t = np.array([2, -100, 5, 0])
    dloss = np.array([0.5, 1.0, 1.5, 0.25])
    return dict(h=h, W=W, b=b, t=t, dloss=dloss, logit_scale=0.75, softcap=4.0)


def main():
    c = case()
    out = {"inputs": {k: (v.tolist() if hasattr(v, "tolist") else v) for k, v in c.items()}}
    kw = dict(logit_scale=c["logit_scale"], softcap=c["softcap"])
    for red in ("mean", "sum", "none"):
        dl = c["dloss"] if red == "none" else np.array([1.0])
        f = oracle.forward(c["h"], c["W"], c["b"], c["t"], reduction=red, **kw)
        g = oracle.backward(c["h"], c["W"], c["b"], c["t"], reduction=red, dloss=dl, **kw)
        out[red] = {
            "loss": np.asarray(f["loss"]).tolist(), "lse": f["lse"].tolist(),
            "entropy": f["entropy"].tolist(), "argmax": f["argmax"].tolist(),
            "correct": f["correct"], "n_valid": f["n_valid"], "entropy_sum": f["entropy_sum"],
            "dh": g["dh"].tolist(), "dW": g["dW"].tolist(), "db": g["db"].tolist(),
        }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1)
        fh.write("\n")


if __name__ == "__main__":
    main()
