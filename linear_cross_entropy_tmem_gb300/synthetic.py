"""Seeded synthetic inputs for the fused linear cross-entropy.

This module only draws random numbers: it holds none of the loss arithmetic, so
both the CUDA library's tests and the CPU oracle can be fed from it.

The workloads mirror the shapes the pages measure on: model heads at 16k tokens
per step (TRL PR #6859, "Benchmark" and "When it is worth turning on" tables),
the single 256-token projection chunk of TRL PR #6863 ("Numbers"), and
Liger-Kernel PR #1574's "every 17th target ignored" recipe ("Details").  No
dataset or trained weight is involved: hidden states are N(0, 1), the head is
N(0, sigma_W), the bias N(0, 0.1), targets uniform in [0, V) with every 17th
position (index % 17 == 16) set to the ignore index, and per-token upstream
gradients U(0, 2) where the reduction is 'none'.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    n_tokens: int
    hidden: int
    vocab: int
    sigma_w: float = 0.02
    hidden_dtype: torch.dtype = torch.bfloat16
    bias: bool = False
    logit_scale: float = 1.0
    softcap: float = 0.0
    reduction: str = "mean"
    ignore_every: int = 17          # 0 = no ignored targets
    ignore_index: int = -100
    seed: int = 0

    def flops(self) -> float:
        """Algorithmic work of one forward+backward: 8*N*V*D (logits, recompute, dh, dW)."""
        return 8.0 * self.n_tokens * self.vocab * self.hidden

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads: a tiny head, a gemma-3-270m-like huge-vocab head, the
# one-chunk projection benchmark, a Qwen3-8B-like head (the headline) and a
# Command-R-like head with every optional feature on.
TINY = Workload("tiny N512 D128 V4096", 512, 128, 4096)
GEMMA = Workload("gemma-3-270m-like N16384 D640 V262144 softcap30", 16384, 640, 262144,
                 softcap=30.0)
CHUNK = Workload("one-chunk N256 D2048 V248320 sum", 256, 2048, 248320,
                 reduction="sum", ignore_every=0)
QWEN8B = Workload("Qwen3-8B-like N16384 D4096 V151936", 16384, 4096, 151936, sigma_w=0.015)
COMMANDR = Workload("Command-R-like N8192 D2048 V128256 fp32-h bias scale softcap none",
                    8192, 2048, 128256, hidden_dtype=torch.float32, bias=True,
                    logit_scale=0.0625, softcap=30.0, reduction="none")

WORKLOADS = {"tiny": TINY, "gemma": GEMMA, "chunk": CHUNK, "qwen8b": QWEN8B,
             "commandr": COMMANDR}


def make_inputs(w: Workload, device="cpu"):
    """Draw (h, W, b, targets, dloss) for a workload, on ``device``.

    The draw uses a ``torch.Generator`` of ``device`` seeded with ``w.seed``,
    so a seed gives the same tensors each time on one kind of device (CPU and
    CUDA generators give different streams).  ``dloss`` is the upstream
    gradient: one element holding 1.0 for mean/sum, U(0, 2) per token for
    'none'.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    kw = dict(generator=g, device=dev, dtype=torch.float32)
    h = torch.randn(w.n_tokens, w.hidden, **kw).to(w.hidden_dtype)
    W = (torch.randn(w.vocab, w.hidden, **kw) * w.sigma_w).to(torch.bfloat16)
    b = None
    if w.bias:
        b = (torch.randn(w.vocab, **kw) * 0.1).to(torch.bfloat16)
    t = torch.randint(0, w.vocab, (w.n_tokens,), generator=g, device=dev, dtype=torch.int64)
    if w.ignore_every > 0:
        t[w.ignore_every - 1::w.ignore_every] = w.ignore_index
    if w.reduction == "none":
        dloss = torch.rand(w.n_tokens, **kw) * 2.0
    else:
        dloss = torch.ones(1, device=dev, dtype=torch.float32)
    return h, W, b, t, dloss
