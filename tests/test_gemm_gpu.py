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


@pytest.fixture
def multicast(request):
    from linear_cross_entropy_tmem_gb300.api import testing_set_multicast
    testing_set_multicast(2 if request.param else 0)
    yield request.param
    testing_set_multicast(1)


@pytest.mark.parametrize("gemm_mode,multicast", [(1, True), (2, False), (2, True)], indirect=True,
                         ids=["single-cta", "cta-pair", "cta-pair-multicast"])
@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 1), (0, 1), (1, 0)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (300, 520, 200), (1, 8, 8), (257, 1000, 1032),
                                   (640, 768, 4096)])
def test_gemm_layouts_match_fp64(lib, gemm_mode, multicast, a_mn, b_mn, M, N, K):
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


@pytest.mark.parametrize("b_mn", [0, 1], ids=["B-K-major", "B-MN-major"])
@pytest.mark.parametrize("M,N,K", [(1100, 768, 1024), (8192, 2048, 512), (513, 256, 64)])
def test_multicast_clusters_are_bitwise_plain_pairs(lib, b_mn, M, N, K):
    """Clusters of two CTA pairs that share the B tile by TMA multicast compute every output element
    with the same MMAs in the same order as plain pairs: the products are bitwise equal, with a
    ragged last 512-row tile (whose second pair may hold no rows at all) and with many units per
    cluster."""
    from linear_cross_entropy_tmem_gb300.api import testing_gemm, testing_set_gemm_mode, testing_set_multicast
    g = torch.Generator().manual_seed(M + N + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    Bm = _store(torch.randn(N, K, generator=g).to(torch.bfloat16), bool(b_mn)).cuda()
    out = {}
    try:
        testing_set_gemm_mode(2)
        for on in (False, True):
            testing_set_multicast(2 if on else 0)
            out[on] = testing_gemm(A, Bm, a_mn_major=False, b_mn_major=bool(b_mn), M=M, N=N, K=K)
            torch.cuda.synchronize()
    finally:
        testing_set_multicast(1)
        testing_set_gemm_mode(0)
    assert torch.equal(out[False], out[True])
    B_nk = Bm.cpu().double() if not b_mn else Bm.cpu().double()[:, :N].T  # logical [N][K]
    ref = A.cpu().double() @ B_nk.T
    assert (out[True].cpu().double() - ref).abs().max().item() <= 2e-5 * K ** 0.5 * 8
