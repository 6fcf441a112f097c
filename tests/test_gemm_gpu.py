"""The tcgen05 GEMM core through the C ABI's test hook: every operand layout the
loss uses (K-major / MN-major A and B), with ragged M, N and K, against an fp64
product of the same bf16 inputs."""
from __future__ import annotations

import pytest
import torch

pytestmark = pytest.mark.gpu


def _store(x: torch.Tensor, mn_major: bool) -> torch.Tensor:
    """x is logical [rows][K]; return storage [rows][K] or [K][rows_padded] (16-byte rows)."""
    if not mn_major:
        return x.contiguous()
    rows, k = x.shape
    pad = (rows + 7) // 8 * 8
    s = torch.zeros(k, pad, dtype=x.dtype)
    s[:, :rows] = x.T
    return s


@pytest.fixture
def gemm_mode(request):
    from linear_cross_entropy_tmem_gb300.api import testing_set_gemm_mode
    testing_set_gemm_mode(request.param)
    yield request.param
    testing_set_gemm_mode(0)


@pytest.mark.parametrize("gemm_mode", [1, 2], indirect=True, ids=["single-cta", "cta-pair"])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 1), (0, 1), (1, 0)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 520, 200), (1, 8, 8), (257, 1000, 1032),
                                   (640, 768, 4096), (1100, 768, 1024), (8192, 2048, 512)])
def test_gemm_layouts_match_fp64(lib, gemm_mode, a_mn, b_mn, M, N, K):
    from linear_cross_entropy_tmem_gb300.api import testing_gemm
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    Bm = torch.randn(N, K, generator=g).to(torch.bfloat16)
    C = testing_gemm(_store(A, a_mn).cuda(), _store(Bm, b_mn).cuda(), a_mn_major=bool(a_mn),
                     b_mn_major=bool(b_mn), M=M, N=N, K=K)
    torch.cuda.synchronize()
    ref = A.double() @ Bm.double().T
    err = (C.cpu().double() - ref).abs().max().item()
    # fp32 accumulation of K products of unit-variance values
    assert err <= 2e-5 * K ** 0.5 * 8, f"max abs err {err}"
