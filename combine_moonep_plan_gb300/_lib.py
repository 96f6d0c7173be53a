"""ctypes binding of libmoonep.so: the C ABI of include/moonep.h, same names.

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  Loading fails loudly when the library is missing; there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoonep.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_BAD_EXPERT = -2
ERR_HIST_MISMATCH = -3
ERR_SLOTS = -4
ERR_CUDA = -5
ERR_DESTROYED = -6
ERR_PLAN = -7
ERR_NOMEM = -8
ERR_TIMEOUT = -9
PLAN_DUP_RECORDS = 1

#: every symbol include/moonep.h declares
EXPORTS = (
    "moonep_query_sizes", "moonep_ctx_create", "moonep_ctx_destroy", "moonep_ctx_free",
    "moonep_ctx_destroyed", "moonep_plan_create", "moonep_plan_destroy",
    "moonep_plan_clone", "moonep_plan", "moonep_dispatch", "moonep_combine",
    "moonep_dispatch_dedup", "moonep_combine_dedup",
    "moonep_prefetch_weight", "moonep_prefetch_rows", "moonep_reduce_redundant_grad", "moonep_hidden_view",
    "moonep_weight_view", "moonep_get_status", "moonep_strerror", "moonep_num_sms",
    "moonep_plan_noalloc", "moonep_prepare", "moonep_plan_rank", "moonep_dispatch_rank",
    "moonep_combine_rank",
)


class MoonepConfig(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int), ("E", ctypes.c_int), ("K", ctypes.c_int),
                ("S", ctypes.c_int), ("H", ctypes.c_int), ("B", ctypes.c_int),
                ("token_padding", ctypes.c_int), ("num_sms", ctypes.c_int)]


_i32p = ctypes.c_void_p


class MoonepCommPlan(ctypes.Structure):
    _fields_ = [("dst", _i32p), ("experts_to_copy", _i32p), ("cu_seqlens", _i32p),
                ("zero_fill_ranges", _i32p), ("remote_stats", _i32p),
                ("dup_counts", _i32p), ("dup_groups", _i32p), ("dup_loffs", _i32p),
                ("internal", _i32p), ("N", ctypes.c_int), ("R", ctypes.c_int),
                ("E", ctypes.c_int), ("B", ctypes.c_int), ("K", ctypes.c_int),
                ("S", ctypes.c_int), ("NvS", ctypes.c_int), ("NvS_padded", ctypes.c_int),
                ("flags", ctypes.c_int), ("internal_bytes", ctypes.c_size_t)]


class MoonepError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} ({code})")


_lib = None


def load(path: str = LIB_PATH):
    """Load libmoonep.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with combine_moonep_plan_gb300.build.build() "
            "(nvcc, sm_103a); there is no CPU fallback")
    lib = ctypes.CDLL(path)
    vp, ci, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    cfgp = ctypes.POINTER(MoonepConfig)
    planp = ctypes.POINTER(MoonepCommPlan)
    sig = {
        "moonep_query_sizes": (ci, [cfgp, ctypes.POINTER(ci), ctypes.POINTER(ci),
                                    ctypes.POINTER(ctypes.c_size_t)]),
        "moonep_ctx_create": (ci, [cfgp, ci, ctypes.POINTER(vp)]),
        "moonep_ctx_destroy": (ci, [vp]),
        "moonep_ctx_free": (None, [vp]),
        "moonep_ctx_destroyed": (ci, [vp]),
        "moonep_num_sms": (ci, [vp]),
        "moonep_plan_create": (ci, [vp, ci, planp]),
        "moonep_plan_destroy": (ci, [planp]),
        "moonep_plan_clone": (ci, [planp, planp, vp]),
        "moonep_plan": (ci, [vp, vp, vp, planp, vp]),
        "moonep_dispatch": (ci, [vp, planp, vp, vp, vp, vp, vp]),
        "moonep_combine": (ci, [vp, planp, vp, vp, vp, vp, vp]),
        "moonep_dispatch_dedup": (ci, [vp, planp, vp, vp, vp, vp, vp]),
        "moonep_combine_dedup": (ci, [vp, planp, vp, vp, vp, vp, vp]),
        "moonep_prefetch_weight": (ci, [vp, planp, ci, ctypes.POINTER(vp), i64, vp]),
        "moonep_prefetch_rows": (ci, [vp, planp, ci, ctypes.POINTER(vp), ctypes.POINTER(i64), vp]),
        "moonep_prepare": (ci, [vp, ctypes.POINTER(ctypes.c_int32), vp, vp, vp, vp, vp]),
        "moonep_reduce_redundant_grad": (ci, [vp, planp, ci, ctypes.POINTER(vp),
                                              ctypes.POINTER(vp), i64, vp]),
        "moonep_hidden_view": (vp, [vp, ci]),
        "moonep_weight_view": (vp, [vp, ci]),
        "moonep_get_status": (ci, [vp, ctypes.POINTER(ci), vp]),
        "moonep_strerror": (ctypes.c_char_p, [ci]),
        "moonep_plan_noalloc": (ci, [cfgp] + [vp] * 10),
        "moonep_plan_rank": (ci, [vp, ci, vp, vp, planp, vp]),
        "moonep_dispatch_rank": (ci, [vp, planp, ci, vp, vp, ctypes.POINTER(vp),
                                      ctypes.POINTER(vp), vp]),
        "moonep_combine_rank": (ci, [vp, planp, ci, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                     vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def strerror(code: int) -> str:
    try:
        return load().moonep_strerror(code).decode()
    except Exception:  # library missing: still format the code
        return f"status {code}"


def check(code: int, where: str) -> None:
    if code != OK:
        raise MoonepError(code, where)


def ptr_array(ptrs):
    arr = (ctypes.c_void_p * len(ptrs))(*ptrs)
    return arr
