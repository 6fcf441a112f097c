"""The C-ABI library builds, loads and exports every declared symbol; host-side
validation returns the documented status codes.  CPU only: no kernel runs."""
from __future__ import annotations

import ctypes
import glob
import os
import re

import pytest

from linear_cross_entropy_tmem_gb300 import binding as B
from linear_cross_entropy_tmem_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        names.update(re.findall(r"FLCE_API\s+[\w\s\*]+?\b(flce_\w+)\s*\(", open(h).read()))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"flce_forward", "flce_backward", "flce_workspace_size", "flce_read_device_status",
            "flce_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(B.SIGNATURES), "binding signatures and headers disagree"


def test_abi_version_and_status_strings(lib):
    assert lib.flce_abi_version() == 3
    for code in range(0, 10):
        assert lib.flce_status_string(code).decode() not in ("", "unknown status")
    assert lib.flce_status_string(12345).decode() == "unknown status"


def test_problem_struct_layout_matches_header():
    # int64 x3, int32 x4, float x2, int64, double, uint32 x2 -> 72 bytes, natural alignment
    assert ctypes.sizeof(B.FlceProblem) == 72
    assert B.FlceProblem.ignore_index.offset == 48
    assert B.FlceProblem.num_items_in_batch.offset == 56
    assert B.FlceProblem.flags.offset == 64


def _problem(**kw):
    base = dict(n_tokens=512, hidden=128, vocab=4096, hidden_dtype=B.FLCE_BF16, weight_dtype=B.FLCE_BF16,
                bias_dtype=B.FLCE_BF16, reduction=B.FLCE_RED_MEAN, logit_scale=1.0,
                final_logit_softcapping=0.0, ignore_index=-100)
    base.update(kw)
    return B.FlceProblem(**base)


def _ws(lib, prob, bwd):
    n = ctypes.c_size_t()
    st = lib.flce_workspace_size(ctypes.byref(prob), bwd, ctypes.byref(n))
    return st, n.value


def test_workspace_size_needs_no_gpu_and_never_scales_with_n_times_v(lib):
    for (N, D, V) in [(512, 128, 4096), (16384, 640, 262144), (256, 2048, 248320), (16384, 4096, 151936),
                      (8192, 2048, 128256)]:
        for bwd in (0, 1):
            st, n = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V), bwd)
            assert st == B.FLCE_OK
            assert n > 0
        st, fw = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V), 0)
        st, bw = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, hidden_dtype=B.FLCE_F32), 1)
        # forward: O(N * splits); backward: one bf16 G chunk of at most 1 GiB,
        # its per-tile dbias sums (1/64 of it in fp32 per 128 rows), the fp32 hi/lo
        # split (4 N D bytes at most) and the fp32 dh slots (4 N D bytes each: one per
        # K split, at most 8 once the dh product has 128 tiles of 128 x 256)
        # five 4-byte split records per token, up to 64 splits x 2 epilogue groups (256 splits for
        # a batch of at most 512 tokens), + z[target]
        max_splits = 256 if N <= 512 else 64
        assert fw <= (5 * 4 * max_splits * 2 + 4) * N + (1 << 20)
        slots = 8 if -(-N // 128) * -(-D // 256) >= 128 else 16
        assert bw <= (1 << 30) + (1 << 30) // 64 + (1 + slots) * 4 * N * D + (1 << 20)
        # the G chunk covers at most about half of the vocabulary
        assert bw <= N * (V // 2 + 256) * 2 * (1 + 1 / 32) + 16 * 4 * N * D + 4 * N * D + (1 << 20)
        if N * V >= 1 << 28:
            assert bw < 2 * N * V  # far below a full (tokens x vocab) bf16 buffer
    st, n = _ws(lib, _problem(n_tokens=0), 1)
    assert st == B.FLCE_OK
    # with the recompute backward the fused call's scratch regions overlap: it needs no more
    # than the larger of the two plus the shared part
    rec = B.FLCE_FLAG_BWD_RECOMPUTE
    for kw in (dict(flags=rec), dict(hidden_dtype=B.FLCE_F32, flags=rec),
               dict(flags=B.FLCE_FLAG_COMPACT_VALID | rec)):
        pr = _problem(n_tokens=4096, hidden=1024, vocab=50000, **kw)
        fw, bw, fu = (_ws(lib, pr, k)[1] for k in (0, 1, 2))
        assert max(fw, bw) <= fu <= fw + bw
    assert _ws(lib, _problem(), 3)[0] == B.FLCE_ERR_INVALID_ARG


def test_fp32_terms_workspace(lib):
    """fp32 operands add their bf16 terms: 2 (default) or 3 (FLCE_FLAG_FP32_FULL) copies of N x D for
    the hidden state and of V x D for an fp32 head; bf16 operands are unaffected by the flag."""
    N, D, V = 1024, 512, 8000
    full = B.FLCE_FLAG_FP32_FULL
    for bwd in (0, 1, 2):
        for rec in (B.FLCE_FLAG_BWD_RECOMPUTE, B.FLCE_FLAG_BWD_KEEP_LOGITS):
            base = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, flags=rec), bwd)[1]
            assert _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, flags=rec | full), bwd)[1] == base
            h2 = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, hidden_dtype=B.FLCE_F32, flags=rec), bwd)[1]
            h3 = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, hidden_dtype=B.FLCE_F32, flags=rec | full), bwd)[1]
            w2 = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, hidden_dtype=B.FLCE_F32, weight_dtype=B.FLCE_F32,
                                   flags=rec), bwd)[1]
            w3 = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, hidden_dtype=B.FLCE_F32, weight_dtype=B.FLCE_F32,
                                   flags=rec | full), bwd)[1]
            assert abs((h2 - base) - 2 * N * D * 2) <= 1024
            assert abs((h3 - h2) - N * D * 2) <= 1024
            assert abs((w2 - h2) - 2 * V * D * 2) <= 1024
            assert abs((w3 - h3) - 3 * V * D * 2) <= 1024


def test_keep_logits_workspace(lib):
    """The token-chunked backward keeps fp32 logits + bf16 G for at most half of the tokens (a batch
    of at most 256 tokens is one chunk), the dbias partials of one chunk and an fp32 dbias and dW
    accumulator; the automatic choice keeps logits from D = 1152 up."""
    keep, rec = B.FLCE_FLAG_BWD_KEEP_LOGITS, B.FLCE_FLAG_BWD_RECOMPUTE
    for (N, D, V) in [(16384, 4096, 151936), (16384, 640, 262144), (8192, 2048, 128256), (4096, 1024, 50000),
                      (300, 200, 1000), (257, 136, 777)]:
        ldz = (V + 31) // 32 * 32
        ws = {f: _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, flags=f), 2) for f in (0, keep, rec)}
        assert all(st == B.FLCE_OK for st, _ in ws.values())
        k, r, a = ws[keep][1], ws[rec][1], ws[0][1]
        assert a == (k if D >= 1152 else r)
        half = ((N + 1) // 2 + 255) // 256 * 256
        # kept logits + G and the dbias partials of one chunk, fp32 dbias and dW accumulators, dh
        # K-split slots (at most 16), split records of one chunk
        bound = 6 * min(half, N) * ldz + 4 * ((half + 31) // 32) * ldz + 4 * ldz + 4 * V * D + 16 * 4 * half * D \
            + (5 * 4 * (256 if N <= 512 else 64) * 2 + 8) * half + (1 << 20)
        assert r < k <= bound
        if N * V >= 1 << 28:  # the chunk's kept logits + G stay within the 4 GiB budget (+ one row group)
            assert k - 4 * V * D - 16 * 4 * half * D - 4 * ((half + 31) // 32) * ldz <= (4 << 30) + 6 * 256 * ldz \
                + (5 * 4 * 64 * 2 + 8) * half + (1 << 20)
    # with compaction the layout adds the compaction buffers (row map, targets, hidden copy,
    # compacted lse / upstream grads, chunk row counts), about (4 + 8 + 2 D + 4 + 4) bytes per token
    for (N, D, V) in [(16384, 4096, 151936), (8192, 2048, 128256), (700, 256, 3000)]:
        k = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, flags=keep), 2)[1]
        st, kc = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, flags=keep | B.FLCE_FLAG_COMPACT_VALID), 2)
        assert st == B.FLCE_OK and k < kc <= k + N * (20 + 2 * D) + (1 << 16)
    # a batch of at most 256 tokens is one chunk of its own rows (rounded up to 32): its kept logits
    # and G, no dW accumulator, dh slots and the split records
    for N in (1, 100, 256):
        D, V = 2048, 248320
        ldz = (V + 31) // 32 * 32
        rows = (N + 31) // 32 * 32
        st, k = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, flags=keep), 2)
        assert st == B.FLCE_OK
        assert 6 * rows * ldz < k <= 6 * rows * ldz + 4 * rows * ldz // 32 + 16 * 4 * 256 * D \
            + (5 * 4 * 256 * 2 + 8) * rows + (1 << 20)
        assert k < 4 * V * D  # in particular no fp32 dW accumulator


def test_frozen_head_workspace(lib):
    """A frozen head needs neither the fp32 dweight / dbias accumulators of the token-chunked
    backward (4 V D + 4 V bytes with more than one chunk) nor the dbias partial sums of either
    backward; the rest of the layout is the same, and the flag changes nothing for the forward."""
    keep, rec, frozen = B.FLCE_FLAG_BWD_KEEP_LOGITS, B.FLCE_FLAG_BWD_RECOMPUTE, B.FLCE_FLAG_FROZEN_HEAD
    for (N, D, V) in [(16384, 4096, 151936), (8192, 2048, 128256), (256, 2048, 248320), (700, 256, 3000)]:
        ldz = (V + 31) // 32 * 32
        info = B.FlceTestingPlanInfo()
        assert lib.flce_testing_plan(ctypes.byref(_problem(n_tokens=N, hidden=D, vocab=V, flags=keep)), 2, 152,
                                     ctypes.byref(info)) == B.FLCE_OK
        nc, chunks = info.token_chunk_rows, info.n_chunks
        k = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, flags=keep), 2)[1]
        kf = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, flags=keep | frozen), 2)[1]
        saved = 4 * ((nc + 31) // 32) * ldz + (4 * V * D + 4 * ldz if chunks > 1 else 0)
        assert 0 <= (k - kf) - saved <= 3 * 256, (N, D, V, k - kf, saved)
        r = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, flags=rec), 1)[1]
        rf = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, flags=rec | frozen), 1)[1]
        assert rf < r
        assert _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, flags=frozen), 0) == \
            _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V), 0)


def test_keep_logits_workspace_has_no_tokens_times_vocab_term(lib):
    """With a bias (its partial column sums are the one per-row-tile scratch), N swept from 512 to
    131072 at V = 262144: the kept-logits workspace stays within the 4 GiB logit budget, the fp32 dW
    and dbias accumulators, the scratch of one token chunk (whose rows the budget bounds) and terms
    linear in N (compaction buffers, block sums), with no N * V term."""
    keep = B.FLCE_FLAG_BWD_KEEP_LOGITS
    V, D = 262144, 2048
    ldz = V
    nc_max = max(256, (4 << 30) // (6 * ldz) // 256 * 256)  # rows of a chunk at the logit budget
    sizes = {}
    for N in (512, 2048, 8192, 32768, 131072):
        nc = min(nc_max, ((N + 1) // 2 + 255) // 256 * 256)
        for flags in (keep, keep | B.FLCE_FLAG_COMPACT_VALID):
            st, k = _ws(lib, _problem(n_tokens=N, hidden=D, vocab=V, flags=flags), 2)
            assert st == B.FLCE_OK
            splits = 256 if nc <= 512 else 64
            chunk = 6 * nc * ldz + 4 * ldz * ((nc + 31) // 32) + 16 * 4 * nc * D + (5 * 4 * splits * 2 + 8) * nc
            linear = N * (20 + 2 * D) + 32 * (N // 256 + 1)
            assert k <= chunk + 4 * V * D + 4 * ldz + linear + (1 << 20), (N, flags, k)
            sizes[(N, flags)] = k
    assert 6 * nc_max * ldz <= 4 << 30
    # from 32768 to 131072 tokens (chunks at the budget) only the per-token block sums grow
    assert sizes[(131072, keep)] - sizes[(32768, keep)] < 1 << 20
    assert sizes[(131072, keep | B.FLCE_FLAG_COMPACT_VALID)] - sizes[(32768, keep | B.FLCE_FLAG_COMPACT_VALID)] \
        < 98304 * (20 + 2 * D) + (1 << 20)


@pytest.mark.parametrize("kw,code", [
    (dict(vocab=0), B.FLCE_ERR_INVALID_ARG),
    (dict(n_tokens=-1), B.FLCE_ERR_INVALID_ARG),
    (dict(hidden=4), B.FLCE_ERR_INVALID_ARG),
    (dict(hidden=130), B.FLCE_ERR_MISALIGNED),
    (dict(reduction=7), B.FLCE_ERR_INVALID_ARG),
    (dict(weight_dtype=B.FLCE_F32), B.FLCE_ERR_DTYPE_MISMATCH),
    (dict(weight_dtype=5, hidden_dtype=B.FLCE_F32), B.FLCE_ERR_UNSUPPORTED_DTYPE),
    (dict(hidden_dtype=5), B.FLCE_ERR_UNSUPPORTED_DTYPE),
    (dict(logit_scale=float("nan")), B.FLCE_ERR_INVALID_ARG),
    (dict(num_items_in_batch=-1.0), B.FLCE_ERR_INVALID_ARG),
    (dict(num_items_in_batch=float("inf")), B.FLCE_ERR_INVALID_ARG),
    (dict(flags=32), B.FLCE_ERR_INVALID_ARG),
    (dict(flags=B.FLCE_FLAG_BWD_RECOMPUTE | B.FLCE_FLAG_BWD_KEEP_LOGITS), B.FLCE_ERR_INVALID_ARG),
    (dict(reserved=1), B.FLCE_ERR_INVALID_ARG),
])
def test_problem_validation(lib, kw, code):
    assert _ws(lib, _problem(**kw), 0)[0] == code
    assert _ws(lib, _problem(**kw), 1)[0] == code


def _fake(addr):
    return ctypes.c_void_p(addr)


def test_call_validation_without_gpu(lib):
    """Argument errors are reported before any CUDA call, so no GPU is needed."""
    p = _problem()
    _, ws = _ws(lib, p, 0)
    good = [_fake(0x10000 * (i + 1)) for i in range(12)]
    h, w, b, t, loss, lse, ent, corr, nv, es, wsp = good[:11]
    fwd = lib.flce_forward
    # null weight
    assert fwd(ctypes.byref(p), h, None, None, t, loss, lse, ent, corr, nv, es, wsp, ws, None) == B.FLCE_ERR_INVALID_ARG
    # null loss output
    assert fwd(ctypes.byref(p), h, w, None, t, None, lse, ent, corr, nv, es, wsp, ws, None) == B.FLCE_ERR_INVALID_ARG
    # misaligned hidden / workspace
    assert fwd(ctypes.byref(p), _fake(0x10008), w, None, t, loss, lse, ent, corr, nv, es, wsp, ws, None) \
        == B.FLCE_ERR_MISALIGNED
    assert fwd(ctypes.byref(p), h, w, None, t, loss, lse, ent, corr, nv, es, _fake(0x10080), ws, None) \
        == B.FLCE_ERR_MISALIGNED
    # workspace too small
    assert fwd(ctypes.byref(p), h, w, None, t, loss, lse, ent, corr, nv, es, wsp, ws - 1, None) \
        == B.FLCE_ERR_WORKSPACE_TOO_SMALL
    # bad bias dtype only matters when a bias is passed
    pb = _problem(bias_dtype=9)
    assert fwd(ctypes.byref(pb), h, w, b, t, loss, lse, ent, corr, nv, es, wsp, ws, None) \
        == B.FLCE_ERR_UNSUPPORTED_DTYPE
    bwd = lib.flce_backward
    _, wsb = _ws(lib, p, 1)
    dh, dw, db = good[8], good[9], good[10]
    # bias and dbias must be both present or both absent
    assert bwd(ctypes.byref(p), h, w, b, t, lse, nv, loss, dh, dw, None, wsp, wsb, None) == B.FLCE_ERR_INVALID_ARG
    assert bwd(ctypes.byref(p), h, w, None, t, lse, nv, loss, dh, dw, db, wsp, wsb, None) == B.FLCE_ERR_INVALID_ARG
    assert bwd(ctypes.byref(p), h, w, None, t, lse, nv, loss, dh, dw, None, wsp, wsb - 1, None) \
        == B.FLCE_ERR_WORKSPACE_TOO_SMALL
    # a frozen head takes no dweight / dbias, and every other problem needs dweight
    pf = _problem(flags=B.FLCE_FLAG_FROZEN_HEAD)
    _, wsf = _ws(lib, pf, 1)
    assert bwd(ctypes.byref(pf), h, w, None, t, lse, nv, loss, dh, dw, None, wsp, wsf, None) == B.FLCE_ERR_INVALID_ARG
    assert bwd(ctypes.byref(pf), h, w, b, t, lse, nv, loss, dh, None, db, wsp, wsf, None) == B.FLCE_ERR_INVALID_ARG
    assert bwd(ctypes.byref(p), h, w, None, t, lse, nv, loss, dh, None, None, wsp, wsb, None) == B.FLCE_ERR_INVALID_ARG
    assert bwd(ctypes.byref(pf), h, w, b, t, lse, nv, loss, dh, None, None, wsp, wsf - 1, None) \
        == B.FLCE_ERR_WORKSPACE_TOO_SMALL  # past the argument checks: only the size is left
    assert lib.flce_read_device_status(None, None, None) == B.FLCE_ERR_INVALID_ARG
    assert lib.flce_testing_set_tuning(-1, 0) == B.FLCE_ERR_INVALID_ARG
    assert lib.flce_testing_set_tuning(0, 17) == B.FLCE_ERR_INVALID_ARG
    assert lib.flce_testing_set_tuning(0, 0) == B.FLCE_OK


def test_python_binding_refuses_cpu_tensors():
    """The product path has no CPU fallback: CPU inputs raise."""
    import torch

    import linear_cross_entropy_tmem_gb300 as F
    h = torch.zeros(4, 8, dtype=torch.bfloat16)
    W = torch.zeros(5, 8, dtype=torch.bfloat16)
    t = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(RuntimeError, match="CUDA"):
        F.flce_forward(h, W, t)


def test_oracle_is_not_imported_by_the_product_path():
    """No module of the package imports the oracle."""
    pkg = os.path.join(ROOT, "linear_cross_entropy_tmem_gb300")
    for f in glob.glob(os.path.join(pkg, "**", "*.py"), recursive=True):
        src = open(f).read()
        assert not re.search(r"^\s*(from|import)\s+oracle\b", src, re.M), f


def test_testing_switches_validate_their_arguments(lib):
    """The process-wide test/tuning switches reject out-of-range values and accept every
    documented one (they only store a setting, so no GPU is needed)."""
    assert lib.flce_testing_set_gemm_mode(3) == B.FLCE_ERR_INVALID_ARG
    assert lib.flce_testing_set_gemm_mode(-1) == B.FLCE_ERR_INVALID_ARG
    try:
        for mode in (1, 2, 0):
            assert lib.flce_testing_set_gemm_mode(mode) == B.FLCE_OK
    finally:
        lib.flce_testing_set_gemm_mode(0)
