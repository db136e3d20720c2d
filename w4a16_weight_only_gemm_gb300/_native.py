"""ctypes binding of libw4a16.so (the C ABI declared in include/w4a16.h).

Argument marshalling only: every step of the path runs in the library's
CUDA kernels.  The library must have been built (``build.build()``); if it
is missing the first call raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_LOCK = threading.Lock()
_LIB = None

OK = 0
STATUS_NAMES = {
    0: "W4A16_OK", 1: "W4A16_ERR_NULL", 2: "W4A16_ERR_SHAPE", 3: "W4A16_ERR_ALIGN",
    4: "W4A16_ERR_CUDA", 5: "W4A16_ERR_TIMEOUT", 6: "W4A16_ERR_DEVICE",
}

# name -> (restype, argtypes); mirrors include/w4a16.h
_P, _I64, _I32, _U64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64
SIGNATURES = {
    "w4a16_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "w4a16_version": (ctypes.c_int, []),
    "w4a16_quantize": (ctypes.c_int, [_P, _I64, _I64, _I32, _P, _P, _P]),
    "w4a16_quantize_ex": (ctypes.c_int, [_P, _I64, _I64, _I32, _I32, _P, _P, _P, _P]),
    "w4a16_repacked_bytes": (_I64, [_I64, _I64]),
    "w4a16_repack": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
    "w4a16_unrepack": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
    "w4a16_gemm": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "w4a16_quantize_q4_0": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
    "w4a16_gemm_q4_0": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I64, _P]),
    "w4a16_quantize_w8": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P]),
    "w4a16_gemm_w8": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "w4a16_gemm_ex": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _P]),
    "w4a16_gemm_plan": (ctypes.c_int, [_I64, _I64, _I64] + [ctypes.POINTER(ctypes.c_int)] * 5),
    "w4a16_gemm_plan_tail": (ctypes.c_int, [_I64, _I64, _I64] + [ctypes.POINTER(ctypes.c_int)] * 2),
    "w4a16_gemm_ex_plan": (ctypes.c_int, [_I64, _I64, _I64, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_int32] + [ctypes.POINTER(ctypes.c_int)] * 4),
    "w4a16_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int)]),
    "w4a16_set_wait_timeout_ns": (None, [_U64]),
    "w4a16_selftest_wait_timeout": (ctypes.c_int, [_U64, _P]),
}


class W4A16Error(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """The loaded library (loaded once; raises if it has not been built)."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build the CUDA library first "
                    "(w4a16_weight_only_gemm_gb300.build.build()); there is no fallback")
            handle = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _LIB = handle
    return _LIB


def check(code: int, where: str) -> None:
    if code != OK:
        raise W4A16Error(code, where)
