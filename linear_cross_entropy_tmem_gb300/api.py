"""Torch-facing calls with the C ABI's names: argument marshalling only.

PyTorch provides device memory (outputs, workspace) and the current CUDA
stream; every step of the loss runs in ``libflce.so``.  Inputs must already be
CUDA tensors: there is no CPU path.
"""
from __future__ import annotations

import ctypes
from typing import NamedTuple, Optional

import torch

from . import binding as B


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None or t.numel() == 0 else ctypes.c_void_p(t.data_ptr())


def _dtype_code(dt: torch.dtype, what: str) -> int:
    if dt == torch.bfloat16:
        return B.FLCE_BF16
    if dt == torch.float32:
        return B.FLCE_F32
    raise TypeError(f"{what}: dtype {dt} is not supported (bf16 or fp32)")


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def make_problem(n_tokens: int, hidden: int, vocab: int, *, hidden_dtype=torch.bfloat16,
                 weight_dtype=torch.bfloat16, bias_dtype=torch.bfloat16, logit_scale: float = 1.0,
                 softcap: float = 0.0, ignore_index: int = -100, reduction: str = "mean",
                 num_items_in_batch: float = 0.0, compact: bool = False,
                 bwd: str = "auto", fp32_full: bool = False, frozen_head: bool = False) -> B.FlceProblem:
    """``bwd`` picks the backward algorithm of the fused call: "auto", "recompute" or
    "keep_logits" (token-chunked; see FLCE_FLAG_BWD_KEEP_LOGITS in include/flce.h).
    ``fp32_full`` splits fp32 operands into three bf16 terms (FLCE_FLAG_FP32_FULL).
    ``frozen_head``: the backward forms dhidden only (FLCE_FLAG_FROZEN_HEAD)."""
    if reduction not in B.REDUCTIONS:
        raise ValueError(f"reduction must be one of {sorted(B.REDUCTIONS)}")
    if bwd not in B.BWD_ALGOS:
        raise ValueError(f"bwd must be one of {sorted(B.BWD_ALGOS)}")
    return B.FlceProblem(
        n_tokens=n_tokens, hidden=hidden, vocab=vocab,
        hidden_dtype=_dtype_code(hidden_dtype, "hidden"), weight_dtype=_dtype_code(weight_dtype, "weight"),
        bias_dtype=_dtype_code(bias_dtype, "bias"), reduction=B.REDUCTIONS[reduction],
        logit_scale=float(logit_scale), final_logit_softcapping=float(softcap), ignore_index=int(ignore_index),
        num_items_in_batch=float(num_items_in_batch),
        flags=(B.FLCE_FLAG_COMPACT_VALID if compact else 0) | B.BWD_ALGOS[bwd]
        | (B.FLCE_FLAG_FP32_FULL if fp32_full else 0) | (B.FLCE_FLAG_FROZEN_HEAD if frozen_head else 0),
        reserved=0)


def flce_workspace_size(problem: B.FlceProblem, for_backward) -> int:
    """Bytes for flce_forward (0 / False), flce_backward (1 / True) or flce_forward_backward (2)."""
    out = ctypes.c_size_t(0)
    B.check(B.load().flce_workspace_size(ctypes.byref(problem), int(for_backward), ctypes.byref(out)),
            "flce_workspace_size")
    return int(out.value)


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise RuntimeError("flce: inputs must be CUDA tensors (the library has no CPU path)")


def _contig(t, name):
    if t is not None and not t.is_contiguous():
        raise ValueError(f"flce: {name} must be contiguous")


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]) -> torch.Tensor:
    if workspace is None:
        return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    if workspace.numel() < nbytes:
        raise ValueError(f"flce: workspace has {workspace.numel()} bytes, needs {nbytes}")
    return workspace


class ForwardResult(NamedTuple):
    loss: torch.Tensor          # [] (mean/sum) or [N] (none), fp32
    lse: torch.Tensor           # [N] fp32
    correct: torch.Tensor       # [] int64
    n_valid: torch.Tensor       # [] int64
    entropy_sum: torch.Tensor   # [] fp32
    entropy: Optional[torch.Tensor]  # [N] fp32 or None
    workspace: torch.Tensor     # holds the device status word


def flce_forward(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor,
                 bias: Optional[torch.Tensor] = None, *, logit_scale: float = 1.0, softcap: float = 0.0,
                 ignore_index: int = -100, reduction: str = "mean", entropy: bool = False,
                 num_items_in_batch: float = 0.0, compact: bool = False,
                 fp32_full: bool = False, workspace: Optional[torch.Tensor] = None) -> ForwardResult:
    """Forward of the fused linear cross-entropy (see ``flce_forward`` in include/flce.h)."""
    _require_cuda(hidden, weight, targets, bias)
    for t, n in ((hidden, "hidden"), (weight, "weight"), (targets, "targets"), (bias, "bias")):
        _contig(t, n)
    if targets.dtype != torch.int64:
        raise TypeError("flce: targets must be int64")
    N, D = hidden.shape
    V = weight.shape[0]
    prob = make_problem(N, D, V, hidden_dtype=hidden.dtype, weight_dtype=weight.dtype,
                        bias_dtype=bias.dtype if bias is not None else torch.bfloat16,
                        logit_scale=logit_scale, softcap=softcap, ignore_index=ignore_index,
                        reduction=reduction, num_items_in_batch=num_items_in_batch, compact=compact,
                        fp32_full=fp32_full)
    dev = hidden.device
    ws = _workspace(flce_workspace_size(prob, False), dev, workspace)
    f32 = dict(dtype=torch.float32, device=dev)
    loss = torch.empty(N if reduction == "none" else 1, **f32)
    lse = torch.empty(N, **f32)
    ent = torch.empty(N, **f32) if entropy else None
    correct = torch.empty(1, dtype=torch.int64, device=dev)
    n_valid = torch.empty(1, dtype=torch.int64, device=dev)
    ent_sum = torch.empty(1, **f32)
    st = B.load().flce_forward(ctypes.byref(prob), _ptr(hidden), _ptr(weight), _ptr(bias), _ptr(targets),
                               _ptr(loss), _ptr(lse), _ptr(ent), _ptr(correct), _ptr(n_valid), _ptr(ent_sum),
                               _ptr(ws), ws.numel(), _stream(dev))
    B.check(st, "flce_forward")
    if reduction != "none":
        loss = loss.view(())
    return ForwardResult(loss, lse, correct.view(()), n_valid.view(()), ent_sum.view(()), ent, ws)


def flce_backward(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor, lse: torch.Tensor,
                  n_valid: torch.Tensor, dloss: torch.Tensor, bias: Optional[torch.Tensor] = None, *,
                  logit_scale: float = 1.0, softcap: float = 0.0, ignore_index: int = -100,
                  reduction: str = "mean", num_items_in_batch: float = 0.0, compact: bool = False,
                  fp32_full: bool = False, frozen_head: bool = False, workspace: Optional[torch.Tensor] = None,
                  outputs=None):
    """Backward (see ``flce_backward`` in include/flce.h); returns (dhidden, dweight, dbias), with
    dweight and dbias None for a frozen head."""
    _require_cuda(hidden, weight, targets, lse, n_valid, dloss, bias)
    for t, n in ((hidden, "hidden"), (weight, "weight"), (targets, "targets"), (bias, "bias"), (lse, "lse")):
        _contig(t, n)
    N, D = hidden.shape
    V = weight.shape[0]
    prob = make_problem(N, D, V, hidden_dtype=hidden.dtype, weight_dtype=weight.dtype,
                        bias_dtype=bias.dtype if bias is not None else torch.bfloat16,
                        logit_scale=logit_scale, softcap=softcap, ignore_index=ignore_index,
                        reduction=reduction, num_items_in_batch=num_items_in_batch, compact=compact,
                        fp32_full=fp32_full, frozen_head=frozen_head)
    dev = hidden.device
    ws = _workspace(flce_workspace_size(prob, True), dev, workspace)
    dloss = dloss.to(dtype=torch.float32).contiguous().reshape(-1)
    n_valid = n_valid.reshape(-1)
    if outputs is None:
        dh = torch.empty_like(hidden)
        dW = torch.empty_like(weight) if not frozen_head else None
        db = torch.empty_like(bias) if bias is not None and not frozen_head else None
    else:
        dh, dW, db = outputs
    st = B.load().flce_backward(ctypes.byref(prob), _ptr(hidden), _ptr(weight), _ptr(bias), _ptr(targets),
                                _ptr(lse), _ptr(n_valid), _ptr(dloss), _ptr(dh), _ptr(dW), _ptr(db), _ptr(ws),
                                ws.numel(), _stream(dev))
    B.check(st, "flce_backward")
    return dh, dW, db


def flce_forward_backward(hidden: torch.Tensor, weight: torch.Tensor, targets: torch.Tensor, dloss: torch.Tensor,
                          bias: Optional[torch.Tensor] = None, *, logit_scale: float = 1.0, softcap: float = 0.0,
                          ignore_index: int = -100, reduction: str = "mean", entropy: bool = False,
                          num_items_in_batch: float = 0.0, compact: bool = False, bwd: str = "auto",
                          fp32_full: bool = False, frozen_head: bool = False,
                          workspace: Optional[torch.Tensor] = None):
    """Forward and backward in one call (see ``flce_forward_backward`` in include/flce.h);
    ``bwd`` as in :func:`make_problem`.

    Returns ``(ForwardResult, (dhidden, dweight, dbias))``, with dweight and dbias None for a frozen
    head."""
    _require_cuda(hidden, weight, targets, dloss, bias)
    for t, n in ((hidden, "hidden"), (weight, "weight"), (targets, "targets"), (bias, "bias")):
        _contig(t, n)
    if targets.dtype != torch.int64:
        raise TypeError("flce: targets must be int64")
    N, D = hidden.shape
    V = weight.shape[0]
    prob = make_problem(N, D, V, hidden_dtype=hidden.dtype, weight_dtype=weight.dtype,
                        bias_dtype=bias.dtype if bias is not None else torch.bfloat16,
                        logit_scale=logit_scale, softcap=softcap, ignore_index=ignore_index,
                        reduction=reduction, num_items_in_batch=num_items_in_batch, compact=compact, bwd=bwd,
                        fp32_full=fp32_full, frozen_head=frozen_head)
    dev = hidden.device
    ws = _workspace(flce_workspace_size(prob, 2), dev, workspace)
    f32 = dict(dtype=torch.float32, device=dev)
    loss = torch.empty(N if reduction == "none" else 1, **f32)
    lse = torch.empty(N, **f32)
    ent = torch.empty(N, **f32) if entropy else None
    correct = torch.empty(1, dtype=torch.int64, device=dev)
    n_valid = torch.empty(1, dtype=torch.int64, device=dev)
    ent_sum = torch.empty(1, **f32)
    dloss = dloss.to(dtype=torch.float32).contiguous().reshape(-1)
    dh = torch.empty_like(hidden)
    dW = torch.empty_like(weight) if not frozen_head else None
    db = torch.empty_like(bias) if bias is not None and not frozen_head else None
    st = B.load().flce_forward_backward(ctypes.byref(prob), _ptr(hidden), _ptr(weight), _ptr(bias), _ptr(targets),
                                        _ptr(dloss), _ptr(loss), _ptr(lse), _ptr(ent), _ptr(correct),
                                        _ptr(n_valid), _ptr(ent_sum), _ptr(dh), _ptr(dW), _ptr(db), _ptr(ws),
                                        ws.numel(), _stream(dev))
    B.check(st, "flce_forward_backward")
    if reduction != "none":
        loss = loss.view(())
    return (ForwardResult(loss, lse, correct.view(()), n_valid.view(()), ent_sum.view(()), ent, ws), (dh, dW, db))


def flce_read_device_status(workspace: torch.Tensor) -> int:
    """Synchronise the current stream and return the device status word of ``workspace``."""
    out = ctypes.c_int(0)
    B.check(B.load().flce_read_device_status(_ptr(workspace), _stream(workspace.device), ctypes.byref(out)),
            "flce_read_device_status")
    return int(out.value)


def flce_status_string(status: int) -> str:
    return B.load().flce_status_string(int(status)).decode()


def scale_gradient(x: torch.Tensor, scale: torch.Tensor) -> torch.Tensor:
    """``x *= scale`` in place on the device (see ``flce_scale_gradient``); ``scale`` is a one-element
    fp32 device tensor, and nothing is read or written when it holds exactly 1."""
    _require_cuda(x, scale)
    _contig(x, "x")
    scale = scale.to(dtype=torch.float32).contiguous().reshape(-1)[:1]
    B.check(B.load().flce_scale_gradient(_ptr(scale), _ptr(x), x.numel(), _dtype_code(x.dtype, "x"),
                                         _stream(x.device)), "flce_scale_gradient")
    return x


class LinearCrossEntropy(torch.autograd.Function):
    """Autograd wrapper: loss of ``hidden @ weight.T (+ bias)`` against ``targets``.

    With ``grad_in_forward`` (the default) and a mean or sum loss, the forward already computes the
    gradients for an upstream gradient of 1 in one fused call (``flce_forward_backward``, which keeps
    the logits of token chunks from D = 1152 up), and the backward scales them by the upstream
    gradient in place (``flce_scale_gradient``; nothing happens for the usual 1).  Gradients are linear
    in a scalar upstream gradient, so this is the same result up to one rounding.  A second backward
    through the same graph recomputes them (``flce_backward``) instead of rescaling.

    When neither the weight nor the bias requires a gradient (a frozen head, e.g. LoRA training),
    only dhidden is formed (``FLCE_FLAG_FROZEN_HEAD``)."""

    @staticmethod
    def forward(ctx, hidden, weight, bias, targets, logit_scale, softcap, ignore_index, reduction,
                num_items_in_batch=0.0, compact=False, grad_in_forward=True, fp32_full=False):
        kw = dict(logit_scale=logit_scale, softcap=softcap, ignore_index=ignore_index, reduction=reduction,
                  num_items_in_batch=num_items_in_batch, compact=compact, fp32_full=fp32_full)
        need = any(ctx.needs_input_grad[:3])
        frozen = not ctx.needs_input_grad[1] and not ctx.needs_input_grad[2]
        ctx.grads = None
        if grad_in_forward and need and reduction != "none":
            ones = torch.ones(1, dtype=torch.float32, device=hidden.device)
            r, grads = flce_forward_backward(hidden, weight, targets, ones, bias, frozen_head=frozen, **kw)
            ctx.grads = grads
        else:
            r = flce_forward(hidden, weight, targets, bias, **kw)
        ctx.save_for_backward(hidden, weight, bias, targets, r.lse, r.n_valid)
        ctx.cfg = dict(kw, frozen_head=frozen)
        ctx.mark_non_differentiable(r.correct, r.n_valid, r.entropy_sum)
        return r.loss, r.correct, r.n_valid, r.entropy_sum

    @staticmethod
    def backward(ctx, dloss, _dc, _dn, _de):
        if ctx.grads is not None:
            dh, dW, db = ctx.grads
            ctx.grads = None  # scaled in place once; another backward recomputes
            g = dloss.reshape(-1)[:1]
            for x in (dh, dW, db):
                if x is not None:
                    scale_gradient(x, g)
        else:
            hidden, weight, bias, targets, lse, n_valid = ctx.saved_tensors
            dh, dW, db = flce_backward(hidden, weight, targets, lse, n_valid, dloss.contiguous(), bias, **ctx.cfg)
        return dh, dW, db, None, None, None, None, None, None, None, None, None


def linear_cross_entropy(hidden, weight, targets, bias=None, *, logit_scale=1.0, softcap=0.0,
                         ignore_index=-100, reduction="mean", num_items_in_batch=0.0, compact=False,
                         grad_in_forward=True, fp32_full=False):
    """Returns (loss, correct, n_valid, entropy_sum); only ``loss`` carries gradients.
    ``grad_in_forward``: see :class:`LinearCrossEntropy`."""
    return LinearCrossEntropy.apply(hidden, weight, bias, targets, float(logit_scale), float(softcap),
                                    int(ignore_index), reduction, float(num_items_in_batch), bool(compact),
                                    bool(grad_in_forward), bool(fp32_full))


def testing_gemm(A: torch.Tensor, B_: torch.Tensor, *, a_mn_major: bool, b_mn_major: bool, M: int, N: int,
                 K: int) -> torch.Tensor:
    """C = A(m,k) B(n,k) through the library's tcgen05 GEMM core (test hook)."""
    C = torch.zeros(M, N, dtype=torch.float32, device=A.device)
    st = B.load().flce_testing_gemm(int(a_mn_major), int(b_mn_major), M, N, K, _ptr(A), A.stride(0), _ptr(B_),
                                    B_.stride(0), _ptr(C), C.stride(0), _stream(A.device))
    B.check(st, "flce_testing_gemm")
    return C


def testing_set_tuning(chunk_cols: int = 0, dh_ksplit: int = 0) -> None:
    B.check(B.load().flce_testing_set_tuning(int(chunk_cols), int(dh_ksplit)), "flce_testing_set_tuning")


def testing_set_token_chunk(rows: int = 0) -> None:
    """Rows per token chunk of the token-chunked backward (0 = automatic; tests and tuning)."""
    B.check(B.load().flce_testing_set_token_chunk(int(rows)), "flce_testing_set_token_chunk")


def testing_set_gemm_mode(mode: int = 0) -> None:
    """0 automatic, 1 single-CTA GEMM kernel only, 2 CTA-pair kernel only (tests, A/B timing)."""
    B.check(B.load().flce_testing_set_gemm_mode(int(mode)), "flce_testing_set_gemm_mode")

