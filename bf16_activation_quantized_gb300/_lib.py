"""ctypes declarations of the C ABI in include/w4a16.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw4a16.so")

_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I = ctypes.c_int
SZ = ctypes.c_size_t


class Options(ctypes.Structure):
    _fields_ = [("arm", I), ("split_k", I), ("tile_tokens", I), ("flags", I)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("arm", I), ("split_k", I), ("tile_tokens", I), ("ctas", I),
                ("workspace_bytes", SZ), ("whole_k", I)]


# name -> (restype, argtypes); mirrors include/w4a16.h one to one.
SIGNATURES = {
    "w4a16_status_string": (ctypes.c_char_p, [I]),
    "w4a16_read_error_word": (I, [ctypes.POINTER(I), I]),
    "w4a16_layout_version": (I, []),
    "w4a16_packed_weight_bytes": (SZ, [I, I]),
    "w4a16_pack_weights": (I, [P, P, I, I, P]),
    "w4a16_plan": (I, [I, I, I, I, ctypes.POINTER(Options), ctypes.POINTER(PlanInfo)]),
    "w4a16_workspace_bytes": (I, [I, I, I, I, ctypes.POINTER(SZ)]),
    "w4a16_gemm": (I, [P, P, P, P, I, I, I, I, P, SZ, P]),
    "w4a16_gemm_ex": (I, [P, P, P, P, I, I, I, I, P, SZ, ctypes.POINTER(Options), P]),
    "w4a16_gemm_partials": (I, [P, P, P, P, I, I, I, I, P, SZ, ctypes.POINTER(Options),
                                ctypes.POINTER(I), P]),
    "w4a16_plan_batched": (I, [I, I, I, I, I, ctypes.POINTER(Options), ctypes.POINTER(PlanInfo)]),
    "w4a16_plan_for_sms": (I, [I, I, I, I, I, I, ctypes.POINTER(Options), ctypes.POINTER(PlanInfo)]),
    "w4a16_gemm_batched": (I, [P, P, P, P, I, I, I, I, I, P, SZ, ctypes.POINTER(Options), P]),
    "w4a16_gemm_zp": (I, [P, P, P, P, P, I, I, I, I, P, SZ, ctypes.POINTER(Options), P]),
    "w4a16_gemm_batched_zp": (I, [P, P, P, P, P, I, I, I, I, I, P, SZ, ctypes.POINTER(Options), P]),
    "w4a16_gemm_grouped_zp": (I, [P, P, P, P, P, P, I, I, I, I, I, P, SZ, P]),
    "w4a16_grouped_workspace_bytes": (I, [I, I, I, I, I, ctypes.POINTER(SZ)]),
    "w4a16_gemm_grouped": (I, [P, P, P, P, P, I, I, I, I, I, P, SZ, P]),
    "w4a16_dequant_fp32": (I, [P, P, P, I, I, I, P]),
    "w4a16_dequant_bf16": (I, [P, P, P, I, I, I, P]),
    "w4a16_dequant_zp_fp32": (I, [P, P, P, P, I, I, I, P]),
    "w4a16_dequant_zp_bf16": (I, [P, P, P, P, I, I, I, P]),
    "w4a16_splitk_reduce": (I, [P, P, I, I, I, P]),
    "w4a16_gemm_noalloc": (I, [P, P, P, P, I, I, I, I, P]),
}


class W4A16Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def lib():
    """The loaded library; raises if it has not been built (there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libw4a16.so not found at {LIB_PATH}: build it with "
                "`python -m bf16_activation_quantized_gb300.build` (no CPU fallback exists)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
        return _lib


def status_string(status: int) -> str:
    return lib().w4a16_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != 0:
        raise W4A16Error(status, where)
