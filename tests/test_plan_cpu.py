"""Host-side planning of the backward (no GPU): the choices flce_testing_plan reports for a device
with a given SM count.  The pinned values are worked out by hand from the planning rules stated in
the library's comments (wave counts of units over 76 CTA pairs of a 152-SM GB300); the grid test
checks the invariants every plan must keep."""
from __future__ import annotations

import ctypes

import pytest

from linear_cross_entropy_tmem_gb300 import binding as B


def _problem(N, D, V, **kw):
    base = dict(n_tokens=N, hidden=D, vocab=V, hidden_dtype=B.FLCE_BF16, weight_dtype=B.FLCE_BF16,
                bias_dtype=B.FLCE_BF16, reduction=B.FLCE_RED_MEAN, logit_scale=1.0,
                final_logit_softcapping=0.0, ignore_index=-100)
    base.update(kw)
    return B.FlceProblem(**base)


def _plan(lib, prob, for_backward, sms=152):
    info = B.FlceTestingPlanInfo()
    st = lib.flce_testing_plan(ctypes.byref(prob), for_backward, sms, ctypes.byref(info))
    assert st == B.FLCE_OK, st
    return info


def cdiv(a, b):
    return -(-a // b)


def test_gemma_like_recompute_plan(lib):
    """N=16384, D=640, V=262144: the G scratch holds 32768 columns (1 GiB of bf16), but 8 chunks of
    128 vocabulary tiles give 8 x 384 dW units = 8 x 6 waves on 76 pairs, while 126-tile chunks
    give 8 x 378 units (5 waves each) plus a 16-tile tail (1 wave): 41 waves.  The dh product has
    64 x 3 = 192 pair tiles; 3 K splits fill 8 waves at 95 %, which beats 1 split (84 %) and
    5 splits (97 %, less 2 % per split)."""
    p = _problem(16384, 640, 262144, final_logit_softcapping=30.0)
    for fb in (1, 2):
        info = _plan(lib, p, fb)
        assert info.keep_logits == 0
        assert info.vocab_chunk_cols == 32768
        assert info.run_chunk_cols == 126 * 256 and info.n_chunks == 9
        assert info.dh_pair == 1 and info.dh_ksplit_max == 6 and info.dh_ksplit == 3


def test_qwen_like_plans(lib):
    """N=16384, D=4096, V=151936.  Fused: kept logits in 4 chunks of 4096 tokens; dh has 16 x 16 =
    256 pair tiles, and 5 K splits (1280 units, 17 waves, 99 %) are the fewest within 1 % of the best
    (8 splits, 99.8 %).  Separate backward: the recompute with 30464-column G chunks run as 30208
    (118 tiles: 5 x 1888 dW units = 5 x 25 waves, plus a 4-tile tail) instead of 5 x 26 waves."""
    p = _problem(16384, 4096, 151936)
    fused = _plan(lib, p, 2)
    assert fused.keep_logits == 1 and fused.token_chunk_rows == 4096 and fused.n_chunks == 4
    assert fused.dh_pair == 1 and fused.dh_ksplit_max == 8 and fused.dh_ksplit == 5
    sep = _plan(lib, p, 1)
    assert sep.keep_logits == 0 and sep.vocab_chunk_cols == 30464
    assert sep.run_chunk_cols == 118 * 256 and sep.n_chunks == 6
    assert sep.dh_ksplit_max == 1 and sep.dh_ksplit == 1


def test_one_chunk_plan(lib):
    """N=256, D=2048, V=248320: the dh product has 8 pair tiles; counted with its up to 16 K splits
    they fill the 76 pairs, so it runs on CTA pairs, and 9 K splits (72 units, 95 % of one wave) win
    (ahead of 8 splits at 84 %); the two 124160-column chunks stay, because a third chunk costs more
    than the one dW wave (K = 256, ~1 us) it would save."""
    info = _plan(lib, _problem(256, 2048, 248320, reduction=B.FLCE_RED_SUM), 1)
    assert info.keep_logits == 0 and info.dh_pair == 1
    assert info.vocab_chunk_cols == 124160 and info.run_chunk_cols == 124160 and info.n_chunks == 2
    assert info.dh_ksplit == 9


def test_one_chunk_fused_plan_keeps_logits(lib):
    """The fused call on the same shape keeps the logits of its one 256-token chunk (D = 2048 >= 1152):
    the dh product over K = V runs on the same 8 pair tiles with 9 K splits.  Its forward has one
    256-row pair tile: 64 vocabulary splits could not fill 76 pairs, so a batch this small may split
    further, and 75 splits of 13 of the 970 vocabulary tiles fill one wave (98.2 %)."""
    info = _plan(lib, _problem(256, 2048, 248320, reduction=B.FLCE_RED_SUM), 2)
    assert info.keep_logits == 1 and info.n_chunks == 1 and info.token_chunk_rows == 256
    assert info.dh_pair == 1 and info.dh_ksplit == 9
    assert (info.fwd_pair, info.fwd_splits, info.fwd_tiles_per_split) == (1, 75, 13)
    small = _plan(lib, _problem(70, 2048, 248320), 2)
    assert small.keep_logits == 1 and small.n_chunks == 1 and small.token_chunk_rows == 96


def test_forward_split_plans(lib):
    """The forward splits the vocabulary so that (m tiles x splits) units fill whole waves of 76
    pairs.  Gemma-like: 64 m tiles x 19 splits of 54 tiles = 1216 units = 16 waves (99.8 % of the
    slots do work); 38 or 57 splits tie and the fewer win.  Qwen3-8B-like, kept logits: each
    4096-token chunk has 16 m tiles, and 33 splits of 18 of its 594 tiles give 528 units in 7 waves
    (99.25 %), ahead of 19 splits of 32 (4 full waves but 97.7 %: the last split is short) and
    46 splits of 13 (96.2 %).  The forward alone (flce_forward) plans the whole batch: 64 m tiles,
    and 33 splits of 18 give 2112 units in 28 waves (99.25 %)."""
    gemma = _problem(16384, 640, 262144, final_logit_softcapping=30.0)
    for fb in (0, 1, 2):
        info = _plan(lib, gemma, fb)
        assert (info.fwd_pair, info.fwd_splits, info.fwd_tiles_per_split) == (1, 19, 54)
    qwen = _problem(16384, 4096, 151936)
    fused = _plan(lib, qwen, 2)
    assert fused.keep_logits == 1
    assert (fused.fwd_pair, fused.fwd_splits, fused.fwd_tiles_per_split) == (1, 33, 18)
    fwd = _plan(lib, qwen, 0)
    assert (fwd.fwd_pair, fwd.fwd_splits, fwd.fwd_tiles_per_split) == (1, 33, 18)
    assert fwd.n_chunks == 0 and fwd.dh_ksplit == 0  # the forward plan only


def test_overrides_apply_to_the_plan(lib):
    try:
        assert lib.flce_testing_set_tuning(1000, 3) == B.FLCE_OK
        info = _plan(lib, _problem(4096, 1024, 50000), 1)
        assert info.vocab_chunk_cols == 1024 and info.run_chunk_cols == 1024
        assert info.n_chunks == cdiv(50000, 1024)
        assert info.dh_ksplit_max == 3 and info.dh_ksplit == 3
    finally:
        lib.flce_testing_set_tuning(0, 0)


def test_plan_rejects_bad_arguments(lib):
    info = B.FlceTestingPlanInfo()
    p = _problem(512, 128, 4096)
    assert lib.flce_testing_plan(ctypes.byref(p), 3, 152, ctypes.byref(info)) == B.FLCE_ERR_INVALID_ARG
    assert lib.flce_testing_plan(ctypes.byref(p), -1, 152, ctypes.byref(info)) == B.FLCE_ERR_INVALID_ARG
    assert lib.flce_testing_plan(ctypes.byref(p), 1, 1, ctypes.byref(info)) == B.FLCE_ERR_INVALID_ARG
    assert lib.flce_testing_plan(ctypes.byref(p), 1, 152, None) == B.FLCE_ERR_INVALID_ARG
    bad = _problem(512, 128, 0)
    assert lib.flce_testing_plan(ctypes.byref(bad), 1, 152, ctypes.byref(info)) != B.FLCE_OK


@pytest.mark.parametrize("sms", [132, 148, 152])
def test_plan_invariants(lib, sms):
    shapes = [(1, 8, 300), (257, 136, 777), (512, 128, 4096), (640, 512, 2560), (1300, 256, 2600),
              (4096, 1024, 50000), (8192, 2048, 128256), (16384, 640, 262144), (3000, 1280, 99999),
              (300, 4096, 151936), (20000, 768, 32000)]
    for N, D, V in shapes:
        for fb in (1, 2):
            info = _plan(lib, _problem(N, D, V), fb, sms)
            assert 1 <= info.dh_ksplit <= info.dh_ksplit_max <= 16
            n_t = cdiv(V, 256)
            fwd_rows = info.token_chunk_rows if info.keep_logits else N
            assert 1 <= info.fwd_splits <= min(256 if fwd_rows <= 512 else 64, n_t)
            assert info.fwd_splits == cdiv(n_t, info.fwd_tiles_per_split)  # no empty split
            if info.keep_logits:
                assert fb == 2 and D >= 1152
                if N > 256:  # at least two chunks: the kept logits never cover the whole batch
                    assert info.token_chunk_rows % 256 == 0
                    assert info.token_chunk_rows <= cdiv(cdiv(N, 2), 256) * 256
                    assert info.n_chunks == cdiv(N, info.token_chunk_rows) >= 2
                else:  # one chunk of the batch's rows, rounded up to 32
                    assert info.token_chunk_rows == cdiv(N, 32) * 32 and info.n_chunks == 1
            else:
                assert fb == 1 or D < 1152
                vc, run = info.vocab_chunk_cols, info.run_chunk_cols
                assert vc % 256 == 0 and run % 256 == 0
                assert run <= vc and run >= max(1, vc // 256 // 2) * 256  # widths down to half the tiles
                assert info.n_chunks == cdiv(V, run)
                assert N * vc * 2 <= max(1 << 30, N * 256 * 2)  # the G chunk stays within 1 GiB


def test_backward_algorithm_follows_flags(lib):
    """The fused call keeps logits from D = 1152 up (a batch of at most 256 tokens as one chunk);
    FLCE_FLAG_BWD_RECOMPUTE and FLCE_FLAG_BWD_KEEP_LOGITS force either algorithm, with and without
    valid-token compaction and fp32 hidden states.  flce_backward always recomputes."""
    rec, keep, cmp_ = B.FLCE_FLAG_BWD_RECOMPUTE, B.FLCE_FLAG_BWD_KEEP_LOGITS, B.FLCE_FLAG_COMPACT_VALID
    for extra in (0, cmp_):
        for dt in (B.FLCE_BF16, B.FLCE_F32):
            kw = dict(hidden_dtype=dt)
            assert _plan(lib, _problem(4096, 1152, 50000, flags=extra, **kw), 2).keep_logits == 1
            assert _plan(lib, _problem(4096, 1024, 50000, flags=extra, **kw), 2).keep_logits == 0
            assert _plan(lib, _problem(4096, 1280, 50000, flags=extra | rec, **kw), 2).keep_logits == 0
            assert _plan(lib, _problem(4096, 640, 50000, flags=extra | keep, **kw), 2).keep_logits == 1
            assert _plan(lib, _problem(256, 4096, 50000, flags=extra | keep, **kw), 2).keep_logits == 1
            assert _plan(lib, _problem(256, 4096, 50000, flags=extra | rec, **kw), 2).keep_logits == 0
            assert _plan(lib, _problem(100, 640, 50000, flags=extra, **kw), 2).keep_logits == 0
            assert _plan(lib, _problem(4096, 4096, 50000, flags=extra | keep, **kw), 1).keep_logits == 0
