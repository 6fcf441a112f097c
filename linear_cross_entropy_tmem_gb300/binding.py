"""ctypes declarations of ``libflce.so`` (the C ABI in ``include/flce.h``).

Loading fails loudly when the library has not been built: there is no
fallback implementation.  Build it with ``__graft_entry__.build()`` or
``python -m linear_cross_entropy_tmem_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libflce.so")

FLCE_F32, FLCE_BF16 = 0, 1
FLCE_RED_NONE, FLCE_RED_SUM, FLCE_RED_MEAN = 0, 1, 2
FLCE_FLAG_COMPACT_VALID = 1
FLCE_FLAG_BWD_RECOMPUTE = 2
FLCE_FLAG_BWD_KEEP_LOGITS = 4
FLCE_FLAG_FP32_FULL = 8
FLCE_FLAG_FROZEN_HEAD = 16
BWD_ALGOS = {"auto": 0, "recompute": FLCE_FLAG_BWD_RECOMPUTE, "keep_logits": FLCE_FLAG_BWD_KEEP_LOGITS}
REDUCTIONS = {"none": FLCE_RED_NONE, "sum": FLCE_RED_SUM, "mean": FLCE_RED_MEAN}

FLCE_OK = 0
FLCE_ERR_INVALID_ARG = 1
FLCE_ERR_UNSUPPORTED_DTYPE = 2
FLCE_ERR_DTYPE_MISMATCH = 3
FLCE_ERR_MISALIGNED = 4
FLCE_ERR_WORKSPACE_TOO_SMALL = 5
FLCE_ERR_CUDA = 6
FLCE_ERR_TARGET_OUT_OF_RANGE = 7
FLCE_ERR_TIMEOUT = 8
FLCE_ERR_UNSUPPORTED_DEVICE = 9


class FlceLaunchRecord(ctypes.Structure):
    """Mirror of ``flce_launch_record``."""
    _fields_ = [("begin_event", c_void_p), ("end_event", c_void_p), ("kind", c_int32), ("reserved", c_int32)]


LAUNCH_KINDS = {0: "fwd_logits", 1: "bwd_recompute", 2: "bwd_dweight", 3: "bwd_dhidden", 4: "other",
                5: "bwd_logit_grad"}


class FlceProblem(ctypes.Structure):
    """Mirror of ``flce_problem``."""
    _fields_ = [
        ("n_tokens", c_int64),
        ("hidden", c_int64),
        ("vocab", c_int64),
        ("hidden_dtype", c_int32),
        ("weight_dtype", c_int32),
        ("bias_dtype", c_int32),
        ("reduction", c_int32),
        ("logit_scale", c_float),
        ("final_logit_softcapping", c_float),
        ("ignore_index", c_int64),
        ("num_items_in_batch", ctypes.c_double),
        ("flags", ctypes.c_uint32),
        ("reserved", ctypes.c_uint32),
    ]


_LIB = None

# name -> (restype, argtypes); every function ``include/*.h`` declares.
class FlceTestingPlanInfo(ctypes.Structure):
    """Mirror of ``flce_testing_plan_info``."""
    _fields_ = [
        ("keep_logits", c_int32),
        ("dh_pair", c_int32),
        ("token_chunk_rows", c_int64),
        ("vocab_chunk_cols", c_int64),
        ("run_chunk_cols", c_int64),
        ("n_chunks", c_int64),
        ("dh_ksplit_max", c_int32),
        ("dh_ksplit", c_int32),
        ("fwd_pair", c_int32),
        ("fwd_splits", c_int32),
        ("fwd_tiles_per_split", c_int32),
        ("reserved", c_int32),
    ]


SIGNATURES = {
    "flce_workspace_size": (c_int, [POINTER(FlceProblem), c_int, POINTER(c_size_t)]),
    "flce_forward": (c_int, [POINTER(FlceProblem), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "flce_backward": (c_int, [POINTER(FlceProblem), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                              c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "flce_forward_backward": (c_int, [POINTER(FlceProblem), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                      c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                      c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "flce_forward_noalloc": (c_int, [POINTER(FlceProblem), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "flce_read_device_status": (c_int, [c_void_p, c_void_p, POINTER(c_int)]),
    "flce_status_string": (c_char_p, [c_int]),
    "flce_abi_version": (c_int, []),
    "flce_testing_set_tuning": (c_int, [c_int64, c_int]),
    "flce_scale_gradient": (c_int, [c_void_p, c_void_p, c_int64, c_int32, c_void_p]),
    "flce_testing_set_gemm_mode": (c_int, [c_int]),
    "flce_testing_plan": (c_int, [POINTER(FlceProblem), c_int, c_int, POINTER(FlceTestingPlanInfo)]),
    "flce_testing_set_token_chunk": (c_int, [c_int64]),
    "flce_testing_set_launch_log": (c_int, [c_void_p, c_int32, POINTER(c_int32)]),
    "flce_testing_launch_count": (c_int64, []),
    "flce_testing_gemm": (c_int, [c_int, c_int, c_int64, c_int64, c_int64, c_void_p, c_int64, c_void_p, c_int64,
                                  c_void_p, c_int64, c_void_p]),
}


def load(path: str = LIB_PATH):
    """Load ``libflce.so`` once and declare every exported function."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(
            f"libflce.so not found at {path}: build it with __graft_entry__.build() "
            "(the CUDA library is required; there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


class FlceError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        lib = load()
        msg = lib.flce_status_string(status).decode()
        super().__init__(f"{where}: FLCE status {status} ({msg})" if where else f"FLCE status {status} ({msg})")
        self.status = status


def check(status: int, where: str = "") -> None:
    if status != FLCE_OK:
        raise FlceError(status, where)
