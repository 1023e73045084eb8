"""ctypes view of ``libtaco.so`` (the C ABI declared in include/taco.h).

There is no fallback: if the library cannot be loaded, every call raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

TACO_OK = 0
STATUS_NAMES = {0: "TACO_OK", 1: "TACO_ERR_INVALID_ARG", 2: "TACO_ERR_UNSUPPORTED",
                3: "TACO_ERR_MISALIGNED", 4: "TACO_ERR_CUDA"}

# name -> (restype, argtypes); mirrors include/taco.h
_P = ctypes.c_void_p
_I64, _I32, _F32, _U64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_uint64
_PP = ctypes.POINTER(ctypes.c_void_p)
SIGNATURES = {
    "taco_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "taco_abi_version": (ctypes.c_int, []),
    "taco_block_supported": (ctypes.c_int, [_I32]),
    "taco_compress": (ctypes.c_int, [_P, _I64, _I64, _I32, _F32, _F32, _P, _P, _P, _P]),
    "taco_decompress": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I32, _P, _I32, _P]),
    "taco_compress_int8": (ctypes.c_int, [_P, _I64, _I64, _I32, _F32, _F32, _P, _P, _P, _P]),
    "taco_decompress_int8": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I32, _P, _I32, _P]),
    "taco_reduce_shards": (ctypes.c_int, [_I32, _PP, _PP, _PP, _I64, _I64, _I32, _F32, _F32,
                                          _P, _P, _P, _P]),
    "taco_reduce_decompress": (ctypes.c_int, [_I32, _PP, _PP, _PP, _I64, _I64, _I32, _F32, _F32,
                                              _P, _P, _P, _P, _I32, _P]),
    "agoq_fp8_accumulate": (ctypes.c_int, [_P, _P, _P, _I64, _I32, _P]),
    "agoq_reduce_shards": (ctypes.c_int, [_I32, _PP, _PP, _I64, _I32, _P, _P, _P]),
    "agoq_laaq_quantize": (ctypes.c_int, [_P, _I64, _I32, _I32, _P, _P, _P]),
    "agoq_laaq_dequantize": (ctypes.c_int, [_P, _P, _I64, _I32, _I32, _P, _I32, _P]),
    "agoq_laaq_dequantize_silu": (ctypes.c_int, [_P, _P, _I64, _I32, _I32, _P, _I32, _P]),
    "agoq_laaq_dequantize_rmsnorm": (ctypes.c_int, [_P, _P, _I64, _I64, _I32, _I32, _P, _F32, _P, _I32, _P]),
    "taco_e4m3_encode": (ctypes.c_int, [_P, _I64, _P, _P]),
    "taco_gemm_compress": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _I32, _F32, _F32, _P, _P, _P, _P, _P, _U64,
                                          _P]),
    "agoq_gemm_accumulate": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _U64, _P]),
    "agoq_gemm_laaq_quantize": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _U64, _P]),
    "taco_gemm_workspace_bytes": (ctypes.c_int, [_I64, _I64, _I64, _P]),
    "taco_host_pipeline_create": (ctypes.c_int, [_I32, _I64, _I64, _I32, _I32, _I32,
                                                 ctypes.POINTER(ctypes.c_void_p),
                                                 ctypes.POINTER(ctypes.c_uint64)]),
    "taco_host_pipeline_run": (ctypes.c_int, [_P, _P, _P, _P, _F32, _F32, _P]),
    "taco_host_pipeline_destroy": (ctypes.c_int, [_P]),
    "taco_two_shot_host_noalloc": (ctypes.c_int, [_I32, _I64, _I64, _I32, _P, _P, _F32, _F32, _P]),
    "taco_watchdog_selftest": (ctypes.c_int, [_P]),
    "taco_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), _I32]),
}


class TacoError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libtaco.so (building it first when it is missing or stale and
    nvcc is available).  Raises if it cannot be loaded."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if build_if_missing:
            try:
                path = _build.build()
            except RuntimeError:
                if not os.path.exists(path):
                    raise
        if not os.path.exists(path):
            raise RuntimeError(f"libtaco.so not found at {path}; run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def check(fn: str, status: int) -> None:
    if status != TACO_OK:
        raise TacoError(fn, status)


def ptr_array(ptrs):
    arr = (ctypes.c_void_p * len(ptrs))(*ptrs)
    return ctypes.cast(arr, _PP), arr
