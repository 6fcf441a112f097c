"""Plain fp64 CPU oracle for fused linear cross-entropy (forward and backward).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the tests, the smoke check in ``__graft_entry__`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code with the CUDA library (no kernels, headers, helpers or
constants) and does not import it.

What it computes is the plain definition of the loss the pages describe, written
out in float64 with NumPy, one step per line, with no blocking, fusion or
reordering beyond applying the per-token definition to a chosen subset of
tokens:

* the logit chain is the one the review of TRL PR #6859 ("Add loss_type="cce",
  a fused linear cross-entropy loaded from the Hub", review by albertvillanova,
  the list of things "verified", bullet 2) checked against the chunked path:
  the product ``hidden @ lm_head.T`` accumulated in at least fp32, then
  ``+ bias``, then ``* logit_scale``, then the final-logit soft cap;
* the entropy metric is ``lse - sum(p * logit)`` on the same logits (same
  bullet), and the accuracy metric is the argmax of those logits;
* ignored positions (``ignore_index``, -100) only zero the per-token weight
  after the product (same review, "Correctness" item 2);
* the per-token loss is kept in a wide type (Liger-Kernel PR #1574, Summary
  item 1) and the none-reduction backward scales each token's gradient by its
  own upstream gradient (same PR, Summary item 2);
* an all-ignored batch gives loss 0 and zero gradients (TRL PR #6859 review,
  "Correctness" item 5 and "Test coverage" item 10).

Inputs are taken exactly as given: bf16 or fp32 arrays are widened to float64
without rounding, so the oracle runs "on the same bf16-rounded inputs" the GPU
receives, and the logits are never rounded to bf16.

Readings where the pages are silent (each also listed in the design notes):

* argmax ties go to the lowest vocabulary index;
* ignored tokens still get an lse and a per-token entropy (every row is swept,
  review "Correctness" item 2), but contribute nothing to the loss, the
  correct count, the entropy sum or n_valid;
* a soft cap ``c <= 0`` means "off"; the bias, when present, is added in wide
  precision after the product;
* the mean divides by the number of valid tokens, and is 0 when there are none;
* a target outside ``[0, V)`` that is not ``ignore_index`` is an error: the
  token is treated as ignored and ``status`` reports it.
"""
from __future__ import annotations

import math

import numpy as np

# Status value the oracle reports when a target is neither ignore_index nor a
# valid vocabulary index (same meaning as the library's device status word).
STATUS_OK = 0
STATUS_TARGET_OUT_OF_RANGE = 1


def widen(x) -> np.ndarray:
    """Exact widening of a float array (NumPy or torch, bf16/fp16/fp32/fp64) to float64."""
    if hasattr(x, "detach"):  # a torch tensor: every bf16/fp32 value is exact in fp64
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def _targets(t) -> np.ndarray:
    if hasattr(t, "detach"):
        t = t.detach().to("cpu").numpy()
    return np.asarray(t, dtype=np.int64)


def logits(h, W, b=None, *, logit_scale=1.0, softcap=0.0) -> np.ndarray:
    """Logit chain of the fused head, in float64.

    TRL PR #6859, review, "verified" bullet 2: matmul, then ``+ bias``, then
    ``* logit_scale``, then soft cap ``c * tanh(x / c)``.  The product is exact
    fp64 here (the kernel's fp32 accumulation is within rounding of it).
    """
    h = widen(h)
    W = widen(W)
    acc = h @ W.T
    x = acc if b is None else acc + widen(b)[None, :]
    x = x * float(logit_scale)
    if softcap > 0.0:
        c = float(softcap)
        return c * np.tanh(x / c)
    return x


def _logsumexp_rows(z: np.ndarray) -> np.ndarray:
    m = z.max(axis=1)
    return m + np.log(np.exp(z - m[:, None]).sum(axis=1))


def forward(h, W, b=None, targets=None, *, logit_scale=1.0, softcap=0.0,
            ignore_index=-100, reduction="mean", num_items_in_batch=0.0) -> dict:
    """Forward of the fused linear cross-entropy: the 4-tuple plus per-token values.

    TRL PR #6859, "What it supports": the helper returns the same 4-tuple as the
    chunked path (loss, and from the same pass the accuracy and the entropy).
    Returned keys:

    ``loss``        scalar (mean / sum) or [N] (none, 0 at ignored tokens)
    ``loss_tok``    [N] per-token loss, 0 at ignored tokens
    ``lse``         [N] log-sum-exp of the transformed logits (every token)
    ``entropy``     [N] ``lse - sum(p * z)`` (every token)
    ``argmax``      [N] lowest index of the largest transformed logit
    ``correct``     count of valid tokens whose argmax equals the target
    ``n_valid``     count of tokens whose target is not ignore_index
    ``entropy_sum`` sum of the per-token entropy over valid tokens
    ``status``      STATUS_OK or STATUS_TARGET_OUT_OF_RANGE

    ``num_items_in_batch`` > 0 replaces n_valid as the mean's denominator (the
    count of valid tokens over a whole accumulated batch; TRL PR #6859 review,
    "Test coverage" item 10, test_num_items_in_batch_reduction).
    """
    if reduction not in ("mean", "sum", "none"):
        raise ValueError(f"reduction must be mean, sum or none, not {reduction!r}")
    t = _targets(targets)
    z = logits(h, W, b, logit_scale=logit_scale, softcap=softcap)
    n_tok, vocab = z.shape

    lse = _logsumexp_rows(z)
    p = np.exp(z - lse[:, None])
    entropy = lse - (p * z).sum(axis=1)          # = -sum p log p (review bullet 2)
    argmax = z.argmax(axis=1)                     # NumPy returns the first maximum

    in_range = (t >= 0) & (t < vocab)
    bad = (t != ignore_index) & ~in_range
    valid = in_range & (t != ignore_index)
    rows = np.arange(n_tok)
    z_t = np.where(valid, z[rows, np.where(valid, t, 0)], 0.0)
    loss_tok = np.where(valid, lse - z_t, 0.0)

    n_valid = int(valid.sum())
    correct = int((valid & (argmax == t)).sum())
    entropy_sum = float(entropy[valid].sum())
    total = float(loss_tok.sum())
    if reduction == "sum":
        loss = total
    elif reduction == "mean":
        denom = float(num_items_in_batch) if num_items_in_batch > 0 else n_valid
        loss = total / denom if denom > 0 else 0.0
    else:
        loss = loss_tok.copy()
    return {
        "loss": loss, "loss_tok": loss_tok, "lse": lse, "entropy": entropy,
        "argmax": argmax, "correct": correct, "n_valid": n_valid,
        "entropy_sum": entropy_sum, "valid": valid,
        "status": STATUS_TARGET_OUT_OF_RANGE if bad.any() else STATUS_OK,
    }


def token_weights(targets, vocab, *, reduction="mean", dloss=1.0, ignore_index=-100,
                  n_valid=None, num_items_in_batch=0.0) -> np.ndarray:
    """Per-token weight ``w_n`` that multiplies the softmax gradient.

    mean: ``g / n_valid`` (0 when n_valid is 0); sum: ``g``; none: ``dloss[n]``
    (Liger-Kernel PR #1574, Summary item 2: each row scaled by its own upstream
    gradient).  Ignored tokens get 0 (TRL PR #6859 review, "Correctness" item 2).
    ``n_valid`` may be given for a subset of tokens whose mean runs over more;
    ``num_items_in_batch`` > 0 replaces it as the mean's denominator.
    """
    t = _targets(targets)
    valid = (t >= 0) & (t < vocab) & (t != ignore_index)
    if n_valid is None:
        n_valid = int(valid.sum())
    if num_items_in_batch > 0:
        n_valid = float(num_items_in_batch)
    if reduction == "none":
        g = widen(dloss).reshape(-1)
        if g.shape[0] != t.shape[0]:
            raise ValueError("reduction='none' needs one upstream gradient per token")
        w = g.copy()
    else:
        g = float(np.asarray(widen(dloss)).reshape(-1)[0])
        if reduction == "sum":
            w = np.full(t.shape[0], g)
        elif reduction == "mean":
            w = np.full(t.shape[0], g / n_valid if n_valid > 0 else 0.0)
        else:
            raise ValueError(reduction)
    return np.where(valid, w, 0.0)


def grad_logits(h, W, b=None, targets=None, *, logit_scale=1.0, softcap=0.0,
                ignore_index=-100, reduction="mean", dloss=1.0, lse=None,
                n_valid=None, vocab_rows=None, num_items_in_batch=0.0) -> np.ndarray:
    """``G = dL/d(acc)``: ``w_n (softmax - onehot) * s * (1 - (z/c)^2)``.

    The derivative of ``c*tanh(s*(acc+b)/c)`` with respect to ``acc`` is
    ``s * (1 - tanh^2) = s * (1 - (z/c)^2)``; without a soft cap it is ``s``.
    ``lse`` may be passed so that a subset of vocabulary columns
    (``vocab_rows``) is evaluated without the other columns; it must then be
    the oracle's own full-vocabulary lse for these tokens.
    """
    t = _targets(targets)
    Wf = widen(W)
    vocab = Wf.shape[0]
    cols = np.arange(vocab) if vocab_rows is None else np.asarray(vocab_rows)
    bb = None if b is None else widen(b)[cols]
    z = logits(h, Wf[cols], bb, logit_scale=logit_scale, softcap=softcap)
    if lse is None:
        if vocab_rows is not None:
            raise ValueError("a vocabulary subset needs the full-vocabulary lse")
        lse = _logsumexp_rows(z)
    p = np.exp(z - np.asarray(lse, dtype=np.float64)[:, None])
    onehot = (t[:, None] == cols[None, :]).astype(np.float64)
    w = token_weights(t, vocab, reduction=reduction, dloss=dloss,
                      ignore_index=ignore_index, n_valid=n_valid, num_items_in_batch=num_items_in_batch)
    dz_dacc = float(logit_scale) * ((1.0 - (z / float(softcap)) ** 2) if softcap > 0.0 else 1.0)
    return w[:, None] * (p - onehot) * dz_dacc


def backward(h, W, b=None, targets=None, *, logit_scale=1.0, softcap=0.0,
             ignore_index=-100, reduction="mean", dloss=1.0, num_items_in_batch=0.0) -> dict:
    """Backward: ``dh = G W``, ``dW = G^T h``, ``db = sum_n G`` (float64, G unrounded).

    TRL PR #6859 review, "Correctness" item 2: the weight gradient is the
    product of the logit gradient's transpose with the hidden states, over every
    token; the hidden gradient is the logit gradient times the head.
    """
    hf = widen(h)
    Wf = widen(W)
    G = grad_logits(hf, Wf, b, targets, logit_scale=logit_scale, softcap=softcap,
                    ignore_index=ignore_index, reduction=reduction, dloss=dloss,
                    num_items_in_batch=num_items_in_batch)
    return {
        "dh": G @ Wf,
        "dW": G.T @ hf,
        "db": None if b is None else G.sum(axis=0),
    }


def forward_rows(h, W, b, targets, rows, **kw) -> dict:
    """The per-token definition of :func:`forward` applied to a subset of tokens.

    Every per-token output depends only on that token's row, so this is the
    same computation restricted to ``rows`` (reduction forced to 'none').
    """
    rows = np.asarray(rows)
    kw = dict(kw)
    kw["reduction"] = "none"
    return forward(widen(h)[rows], W, b, _targets(targets)[rows], **kw)


def lse_all(h, W, b=None, *, logit_scale=1.0, softcap=0.0, row_block=256) -> np.ndarray:
    """Per-token lse for every token, one group of tokens at a time (per-token definition)."""
    hf = widen(h)
    Wf = widen(W)
    out = np.empty(hf.shape[0])
    for r0 in range(0, hf.shape[0], row_block):
        z = logits(hf[r0:r0 + row_block], Wf, b, logit_scale=logit_scale, softcap=softcap)
        out[r0:r0 + row_block] = _logsumexp_rows(z)
    return out


def dweight_rows(h, W, b, targets, vocab_rows, lse, *, logit_scale=1.0, softcap=0.0,
                 ignore_index=-100, reduction="mean", dloss=1.0, num_items_in_batch=0.0):
    """Rows ``vocab_rows`` of dW and db, given the oracle's own full lse of every token."""
    hf = widen(h)
    G = grad_logits(hf, W, b, targets, logit_scale=logit_scale, softcap=softcap,
                    ignore_index=ignore_index, reduction=reduction, dloss=dloss,
                    lse=lse, vocab_rows=vocab_rows, num_items_in_batch=num_items_in_batch)
    return G.T @ hf, G.sum(axis=0)


def dhidden_rows(h, W, b, targets, rows, *, n_valid, logit_scale=1.0, softcap=0.0,
                 ignore_index=-100, reduction="mean", dloss=1.0, num_items_in_batch=0.0) -> np.ndarray:
    """Rows ``rows`` of dh (each needs only its own token's logits)."""
    rows = np.asarray(rows)
    t = _targets(targets)
    g = widen(dloss).reshape(-1)
    g_rows = g[rows] if reduction == "none" else g[:1]
    G = grad_logits(widen(h)[rows], W, b, t[rows], logit_scale=logit_scale,
                    softcap=softcap, ignore_index=ignore_index, reduction=reduction,
                    dloss=g_rows, n_valid=n_valid, num_items_in_batch=num_items_in_batch)
    return G @ widen(W)


def relative_frobenius(a, ref) -> float:
    """``||a - ref||_F / ||ref||_F`` (0 when both are zero)."""
    a = widen(a)
    ref = widen(ref)
    den = math.sqrt(float((ref * ref).sum()))
    num = math.sqrt(float(((a - ref) ** 2).sum()))
    if den == 0.0:
        return 0.0 if num == 0.0 else math.inf
    return num / den
