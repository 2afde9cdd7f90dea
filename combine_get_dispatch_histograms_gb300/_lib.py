"""ctypes declarations of libep_gb300.so (see include/ep.h).

Loading fails loudly when the library has not been built: there is no CPU or
library fallback for any step of the path.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

P = ctypes.c_void_p
I32 = ctypes.c_int32
I64 = ctypes.c_int64
INT = ctypes.c_int

EP_OK = 0
STATUS = {0: "EP_OK", -1: "EP_ERR_INVALID_ARG", -2: "EP_ERR_INVALID_INPUT", -3: "EP_ERR_CAPACITY",
          -4: "EP_ERR_TIMEOUT", -5: "EP_ERR_CUDA"}


class EpConfig(ctypes.Structure):
    _fields_ = [("num_ranks", I32), ("num_experts", I32), ("num_topk", I32), ("num_tokens", I32),
                ("hidden", I32), ("num_channels", I32), ("num_nodes", I32)]


class EpDispatchHandle(ctypes.Structure):
    _fields_ = [(name, P) for name in (
        "recv_count", "recv_offsets", "num_recv_tokens", "rank_base", "num_recv_per_expert",
        "expert_offsets", "perm_rank_base", "channel_prefix_matrix", "send_pos", "perm_pos",
        "stage_base", "stage_pos")]


# name -> (restype, argtypes); every name here is declared in include/ep.h
SIGNATURES = {
    "ep_last_error": (ctypes.c_char_p, []),
    "ep_status_name": (ctypes.c_char_p, [INT]),
    "ep_version": (ctypes.c_char_p, []),
    "ep_ctx_create": (INT, [ctypes.POINTER(EpConfig), ctypes.POINTER(P)]),
    "ep_ctx_destroy": (None, [P]),
    "ep_ctx_check": (INT, [P, P]),
    "ep_ctx_set_wait_timeout_us": (INT, [P, I64]),
    "ep_ctx_set_expert_alignment": (INT, [P, INT]),
    "ep_ctx_expert_alignment": (I32, [P]),
    "ep_ctx_last_launches": (I32, [P]),
    "ep_get_dispatch_layout": (INT, [P, P, P, P, P, P, P, P]),
    "ep_get_dispatch_layout_noalloc": (INT, [I32, I32, I32, I32, I32, P, P, P, P, P, P, P, P]),
    "ep_notify_dispatch": (INT, [P, P, P, P, P, P, P, ctypes.POINTER(EpDispatchHandle), P, P, P, P]),
    "ep_layout_notify": (INT, [P, P, P, P, P, P, P, ctypes.POINTER(EpDispatchHandle), P, P, P, P]),
    "ep_dispatch": (INT, [P, P, P, P, ctypes.POINTER(EpDispatchHandle), P, P, P, P, P, I64, P]),
    "ep_permute": (INT, [P, ctypes.POINTER(EpDispatchHandle), P, P, P, P, I64, P, P, I64, P]),
    "ep_dispatch_permuted": (INT, [P, P, P, P, ctypes.POINTER(EpDispatchHandle), P, P, P, I64, P]),
    "ep_fp8_row_bytes": (I64, [INT]),
    "ep_quantize_fp8": (INT, [P, P, P, P]),
    "ep_dispatch_fp8": (INT, [P, P, P, P, ctypes.POINTER(EpDispatchHandle), P, P, P, P, P, I64, P]),
    "ep_dispatch_quant": (INT, [P, P, P, P, ctypes.POINTER(EpDispatchHandle), P, P, P, P, P, I64, P]),
    "ep_permute_fp8": (INT, [P, ctypes.POINTER(EpDispatchHandle), P, P, P, P, I64, P, P, I64, P]),
    "ep_dispatch_permuted_fp8": (INT, [P, P, P, P, ctypes.POINTER(EpDispatchHandle), P, P, P, I64, P]),
    "ep_dispatch_permuted_quant": (INT, [P, P, P, P, ctypes.POINTER(EpDispatchHandle), P, P, P, I64, P]),
    "ep_combine": (INT, [P, ctypes.POINTER(EpDispatchHandle), P, I64, P, P, P, P]),
    "ep_dispatch_hier": (INT, [P, P, P, P, ctypes.POINTER(EpDispatchHandle), P, P, P, I64, P, P, P, P, P, I64, P]),
    "ep_combine_hier": (INT, [P, ctypes.POINTER(EpDispatchHandle), P, I64, P, P, P, P]),
    "ep_ll_message_bytes": (I64, [INT]),
    "ep_ll_size_hint": (I64, [INT, INT, INT, INT]),
    "ep_ll_buffer_create": (INT, [ctypes.POINTER(EpConfig), INT, ctypes.POINTER(P)]),
    "ep_ll_buffer_destroy": (None, [P]),
    "ep_ll_set_wait_timeout_us": (INT, [P, I64]),
    "ep_ll_set_wait_trace": (INT, [P, P]),
    "ep_ll_send": (INT, [P, P, P, INT, INT, P, P]),
    "ep_ll_recv": (INT, [P, P, P, P, P, P, P]),
    "ep_ll_dispatch": (INT, [P, P, P, INT, INT, P, P, P, P, P, P, P]),
    "ep_ll_combine": (INT, [P, P, P, P, P, P, INT, INT, P, P]),
    "ep_ll_check": (INT, [P, P]),
    "ep_ll_count_slots": (P, [P, INT]),
    "ep_ll_current_buffer": (INT, [P]),
}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libep_gb300.so (building it with nvcc if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing:
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libep_gb300.so is not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


class EpError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn}: {STATUS.get(code, code)}: {msg}")
        self.code = code
        self.status = STATUS.get(code, str(code))


def check(fn: str, code: int):
    if code != EP_OK:
        msg = load().ep_last_error()
        raise EpError(fn, code, msg.decode() if msg else "")
