"""ctypes binding of libcq.so (argument marshalling only).

The library must have been built (``combine_quant_gb300.build``); loading
fails loudly otherwise. There is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcq.so")

CONFIG_FIELDS = (
    "ep_world_size", "moe_expert_num", "shared_expert_num", "shared_expert_rank_num",
    "zero_expert_num", "copy_expert_num", "const_expert_num", "max_bs", "topk", "hidden",
    "global_bs", "quant_mode", "expert_token_nums_type", "mask_ndim", "x_dtype", "smooth_kind",
    "y_dtype",
)

CQ_OK = 0
CQ_ERR_ARG = -1
CQ_ERR_UNSUPPORTED = -2
CQ_ERR_CUDA = -3
CQ_ERR_WORKSPACE = -4
CQ_ERR_TOO_LARGE = -5
NOALLOC_SCRATCH_BYTES = 4 << 20
CQ_ST_BAD_ID = 1
CQ_ST_BAD_MASK = 2
CQ_ST_INTERNAL = 4
CQ_ST_TIMEOUT = 8
CQ_INV_NONE = -1
CQ_INV_COPY = -2
CQ_INV_CONST_BASE = -3

# Every symbol include/cq.h declares.
EXPORTS = (
    "cq_check_config", "cq_local_expert_num", "cq_num_slots", "cq_max_rows", "cq_scale_cols",
    "cq_assist_info_size", "cq_workspace_size", "cq_dispatch_workspace_size",
    "cq_workspace_init", "cq_dispatch",
    "cq_dispatch_route", "cq_dispatch_permute", "cq_combine", "moe_dispatch", "moe_combine",
    "cq_read_status", "cq_strerror", "cq_dispatch_noalloc", "cq_combine_quant", "cq_combine_q8",
    "cq_read_combine_status", "cq_check_bounded_wait", "cq_combine_ws", "cq_dispatch_one_kernel",
)


class CqConfig(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int32) for f in CONFIG_FIELDS]


class CqError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


_LIB = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libcq.so and declare its signatures (once)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise ImportError(
            f"libcq.so not found at {path}: build it with `python -m combine_quant_gb300.build` "
            "(the CUDA path has no fallback)")
    L = ctypes.CDLL(path)
    P, cfgp = ctypes.c_void_p, ctypes.POINTER(CqConfig)
    i32, i64, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "cq_check_config": ([cfgp], ctypes.c_int),
        "cq_local_expert_num": ([cfgp], i32),
        "cq_num_slots": ([cfgp], i32),
        "cq_max_rows": ([cfgp], i64),
        "cq_scale_cols": ([cfgp], i32),
        "cq_assist_info_size": ([cfgp], i64),
        "cq_workspace_size": ([cfgp], sz),
        "cq_dispatch_workspace_size": ([cfgp], sz),
        "cq_dispatch_one_kernel": ([cfgp, ctypes.c_int], ctypes.c_int),
        "cq_workspace_init": ([P, sz, P], ctypes.c_int),
        "cq_dispatch": ([cfgp] + [P] * 13 + [sz, P], ctypes.c_int),
        "moe_dispatch": ([cfgp] + [P] * 13 + [sz, P], ctypes.c_int),
        "cq_dispatch_route": ([cfgp] + [P] * 7 + [sz, P], ctypes.c_int),
        "cq_dispatch_permute": ([cfgp] + [P] * 11 + [sz, P], ctypes.c_int),
        "cq_combine": ([cfgp] + [P] * 8 + [i32, P, P], ctypes.c_int),
        "moe_combine": ([cfgp] + [P] * 8 + [i32, P, P], ctypes.c_int),
        "cq_combine_ws": ([cfgp] + [P] * 8 + [i32, P, P, sz, P], ctypes.c_int),
        "cq_read_status": ([P, P, P], ctypes.c_int),
        "cq_read_combine_status": ([P, P], ctypes.c_int),
        "cq_check_bounded_wait": ([P, P, P], ctypes.c_int),
        "cq_dispatch_noalloc": ([cfgp] + [P] * 13, ctypes.c_int),
        "cq_combine_quant": ([cfgp] + [P] * 5, ctypes.c_int),
        "cq_combine_q8": ([cfgp] + [P] * 9 + [i32, P, P], ctypes.c_int),
        "cq_strerror": ([ctypes.c_int], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _LIB = L
    return L


def strerror(code: int) -> str:
    try:
        return load().cq_strerror(int(code)).decode()
    except ImportError:
        return "libcq not loaded"


def check(rc: int, what: str) -> None:
    if rc != CQ_OK:
        raise CqError(rc, what)
