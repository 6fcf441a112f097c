"""The bf16 term split of fp32 operands (FLCE_FLAG_FP32_FULL and the default
two-term split), checked on the CPU with torch's round-to-nearest bf16 cast:
t0 = rn(x), t1 = rn(x - t0), t2 = rn(x - t0 - t1).  Three terms reproduce every
fp32 value with |x| >= 2^-100 exactly (closer to the bottom of the fp32 range
the lower terms become subnormal and lose bits); two leave a residual below
2^-16 of |x|.  The GPU
kernels compute the same terms (their parity tests check the products)."""
from __future__ import annotations

import numpy as np
import torch


def _terms(x: torch.Tensor):
    t0 = x.to(torch.bfloat16).float()
    r0 = x - t0            # exact in fp32: t0 is x rounded to 8 significant bits
    t1 = r0.to(torch.bfloat16).float()
    r1 = r0 - t1
    t2 = r1.to(torch.bfloat16).float()
    return t0, t1, t2


def test_three_terms_are_exact_and_two_are_within_2_pow_minus_16():
    g = torch.Generator().manual_seed(0)
    mant = torch.rand(200000, generator=g, dtype=torch.float64) + 1.0
    expo = torch.randint(-100, 100, (200000,), generator=g).double()
    sign = torch.where(torch.rand(200000, generator=g) < 0.5, -1.0, 1.0).double()
    x = (sign * mant * torch.pow(2.0, expo)).float()
    x = torch.cat([x, torch.randn(100000, generator=g), torch.tensor([1.0, -1.0, 3.0e38, 2.0 ** -100, 0.0])])
    t0, t1, t2 = _terms(x)
    xd, s2, s3 = x.double(), (t0.double() + t1.double()), (t0.double() + t1.double() + t2.double())
    assert torch.equal(s3, xd)
    nz = xd != 0
    rel2 = ((s2 - xd).abs()[nz] / xd.abs()[nz]).max().item()
    assert rel2 <= 2.0 ** -16
    # the terms shrink by at least 2^-8 each (so products of total order k are ~2^-8k of the leading one)
    big = t1 != 0
    assert torch.all(t1.abs()[big] <= t0.abs()[big] * 2.0 ** -8)
    assert float(np.log2(rel2)) < -16.5  # and it is not loose by much: about 2^-17
