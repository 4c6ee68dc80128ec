"""ctypes loader of libep_gb300.so (the C ABI of include/ep_api.h).

Argument marshalling only.  There is no fallback: if the library is missing
or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

EP_SUCCESS = 0
EP_ERR_INVALID_ARGS = 3
EP_ERR_NOT_FOUND = 4
EP_ERR_BAD_STATE = 6
EP_ERR_GPU_OP = 7
EP_ERR_TIMEOUT = 8
EP_ERR_CAPACITY = 9
EP_ERR_BAD_INDEX = 10
STATUS_NAMES = {
    0: "EP_SUCCESS", 1: "EP_INIT", 2: "EP_IN_PROGRESS",
    3: "EP_ERR_INVALID_ARGS", 4: "EP_ERR_NOT_FOUND", 5: "EP_ERR_RDMA_OP",
    6: "EP_ERR_BAD_STATE", 7: "EP_ERR_GPU_OP", 8: "EP_ERR_TIMEOUT",
    9: "EP_ERR_CAPACITY", 10: "EP_ERR_BAD_INDEX",
}
EP_DEVERR_BAD_INDEX = 0x1
EP_DEVERR_CAPACITY = 0x2
EP_DEVERR_TIMEOUT = 0x4
EP_DEVERR_COMBINE_MISMATCH = 0x8
EP_DT_BF16, EP_DT_FP8_E4M3, EP_DT_FP32 = 0, 1, 2


class EpConfigC(ctypes.Structure):
    _fields_ = [
        ("world_size", ctypes.c_int32),
        ("num_experts", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("hidden", ctypes.c_int32),
        ("max_tokens_per_rank", ctypes.c_int32),
        ("max_recv_tokens_per_rank", ctypes.c_int32),
        ("dispatch_dtype", ctypes.c_int32),
        ("early_notify", ctypes.c_int32),
        ("fused_recv", ctypes.c_int32),
        ("combine_dtype", ctypes.c_int32),
        ("wait_timeout_ns", ctypes.c_int64),
        ("max_grouped_rows_per_rank", ctypes.c_int32),
        ("combine_mode", ctypes.c_int32),
    ]


class EpMoeOutC(ctypes.Structure):
    _fields_ = [
        ("xg", ctypes.c_void_p),
        ("xg_scales", ctypes.c_void_p),
        ("g_src", ctypes.c_void_p),
        ("g_w", ctypes.c_void_p),
        ("yg", ctypes.c_void_p),
        ("entry_slot", ctypes.c_void_p),
        ("rank_stride_bytes", ctypes.c_int64),
        ("count", ctypes.c_void_p),
        ("offset", ctypes.c_void_p),
        ("gcap", ctypes.c_int32),
        ("experts_per_rank", ctypes.c_int32),
    ]


class EpDispatchOutC(ctypes.Structure):
    _fields_ = [
        ("out", ctypes.c_void_p),
        ("out_scales", ctypes.c_void_p),
        ("out_w", ctypes.c_void_p),
        ("out_idx", ctypes.c_void_p),
        ("src_pos", ctypes.c_void_p),
        ("rank_stride_bytes", ctypes.c_int64),
        ("recv_count", ctypes.c_void_p),
        ("send_counts", ctypes.c_void_p),
        ("pos", ctypes.c_void_p),
        ("dispatch_flags", ctypes.c_void_p),
        ("combine_flags", ctypes.c_void_p),
        ("dispatch_epoch", ctypes.c_uint32),
        ("combine_epoch", ctypes.c_uint32),
        ("cap", ctypes.c_int32),
        ("max_dest", ctypes.c_int32),
        ("combine_stage", ctypes.c_void_p),
    ]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_S = ctypes.c_int

SIGNATURES = {
    "ep_status_str": (ctypes.c_char_p, [_S]),
    "ep_workspace_size": (_S, [ctypes.POINTER(EpConfigC), ctypes.POINTER(ctypes.c_size_t)]),
    "ep_create": (_S, [ctypes.POINTER(EpConfigC), _P, ctypes.c_size_t, ctypes.POINTER(_P)]),
    "ep_destroy": (_S, [_P]),
    "ep_layout": (_S, [_P, _P, _P, _P]),
    "ep_dispatch_send": (_S, [_P, _P, _P, _P, _P, _P, _P]),
    "ep_dispatch_recv": (_S, [_P, _P]),
    "ep_dispatch": (_S, [_P, _P, _P, _P, _P, _P, _P]),
    "ep_dispatch_send_replay": (_S, [_P, _P, _P, _P, _P, _P, _P]),
    "ep_dispatch_outputs": (_S, [_P, ctypes.POINTER(EpDispatchOutC)]),
    "ep_get_combine_input_buffer": (_S, [_P, _I32, ctypes.POINTER(_P), ctypes.POINTER(_I64)]),
    "ep_get_combine_input_scales": (_S, [_P, ctypes.POINTER(_P), ctypes.POINTER(_I64)]),
    "ep_combine_send": (_S, [_P, _P]),
    "ep_combine_recv": (_S, [_P, _P, _I64, _P, _I64, _P, _P, _P, _P]),
    "ep_combine": (_S, [_P, _P, _I64, _P, _I64, _P, _P, _P, _P]),
    "ep_reset": (_S, [_P, _P]),
    "ep_get_error": (_S, [_P, ctypes.POINTER(ctypes.c_uint32), _P]),
    "ep_test_identity_expert": (_S, [_P, _P, _I64, _P]),
    "ep_moe_group": (_S, [_P, _P]),
    "ep_moe_outputs": (_S, [_P, ctypes.POINTER(EpMoeOutC)]),
    "ep_moe_ungroup": (_S, [_P, _P, _I64, _P]),
    "ep_test_fp8_quotient_check": (_S, [_P, _P]),
    "ep_layout_noalloc": (_S, [_I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P]),
}


class EpError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load (building first if needed and possible) and return the library."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing; run "
                               "`python -m combine_ep_layout_06_gb300.build`")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
        return L


def check(status: int, what: str):
    if status != EP_SUCCESS:
        raise EpError(status, what)
