"""bench.py's algorithmic accounting (CPU only): the per-kernel flops and bytes that the roofline
divides by the measured time, checked against hand-worked values for the headline head (kept
logits, four 4096-token chunks) and the one-chunk head."""
from __future__ import annotations

import pytest

import bench
from linear_cross_entropy_tmem_gb300.synthetic import WORKLOADS


def test_headline_kept_logits_accounting():
    w = WORKLOADS["qwen8b"]
    N, D, V = 16384, 4096, 151936
    m = bench.kernel_model(w, True, N, {"bwd_logit_grad": 4}, 1, 1)
    assert set(m) == {"fwd_logits", "bwd_logit_grad", "bwd_dhidden", "bwd_dweight"}
    for k in ("fwd_logits", "bwd_dhidden", "bwd_dweight"):
        assert m[k][0] == 2 * N * V * D
    # forward: h once, the head once per chunk; the fp32 logits written
    assert m["fwd_logits"][1:] == (2 * N * D + 4 * 2 * V * D, 4 * N * V)
    # G from the kept logits: 4 bytes read and 2 written per logit
    assert m["bwd_logit_grad"] == (0.0, 4 * N * V, 2 * N * V)
    # dh: G and the head once per chunk read, dh written
    assert m["bwd_dhidden"][1:] == (2 * N * V + 4 * 2 * V * D, 2 * N * D)
    # dW: G and h read; the fp32 accumulator read by chunks 1-3 and written by chunks 0-2; bf16 dW
    assert m["bwd_dweight"][1:] == (2 * N * V + 2 * N * D + 3 * 4 * V * D, 3 * 4 * V * D + 2 * V * D)
    # every product is tensor-bound at the measured peaks (1.7 PFLOP/s, 6.8 TB/s)
    for k in ("fwd_logits", "bwd_dhidden", "bwd_dweight"):
        fl, rd, wr = m[k]
        assert fl / 1.7e15 > (rd + wr) / 6.8e12 and fl / 1.7e15 > wr / 4.0e12


def test_one_chunk_accounting_is_hbm_bound():
    w = WORKLOADS["chunk"]
    N, D, V = 256, 2048, 248320
    m = bench.kernel_model(w, True, N, {"bwd_logit_grad": 1}, 1, 1)
    # one chunk: no fp32 dW accumulator, dW written once in bf16
    assert m["bwd_dweight"][1:] == (2 * N * V + 2 * N * D, 2 * V * D)
    for k in ("fwd_logits", "bwd_dhidden"):
        fl, rd, wr = m[k]
        assert (rd + wr) / 6.8e12 > fl / 1.9e15  # below the ridge point
    fl, rd, wr = m["bwd_dweight"]
    assert wr / 4.0e12 > (rd + wr) / 6.8e12 > fl / 1.9e15  # the write floor is the largest


@pytest.mark.parametrize("name", ["gemma", "tiny"])
def test_recompute_accounting(name):
    w = WORKLOADS[name]
    N, D, V = w.n_tokens, w.hidden, w.vocab
    m = bench.kernel_model(w, False, N, {"bwd_recompute": 3}, 1, 1)
    assert set(m) == {"fwd_logits", "bwd_recompute", "bwd_dhidden", "bwd_dweight"}
    # the recompute reads h once per vocabulary chunk and writes the bf16 G of every logit
    assert m["bwd_recompute"][1:] == (3 * 2 * N * D + 2 * V * D, 2 * N * V)
    assert m["bwd_dweight"][2] == 2 * V * D
