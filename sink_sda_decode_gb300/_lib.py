"""ctypes loader for libsda.so, with the signatures of include/sda.h.

The library is loaded from this package directory only.  If it is missing or
does not load, every call raises: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsda.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "sda.h")

SDA_OK = 0
STATUS_NAMES = {0: "SDA_OK", 1: "SDA_ERR_INVALID_ARG", 2: "SDA_ERR_UNSUPPORTED", 3: "SDA_ERR_CUDA",
                4: "SDA_ERR_WORKSPACE"}

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int
_f32 = ctypes.c_float

SIGNATURES = {
    "sda_strerror": (ctypes.c_char_p, [_i32]),
    "sda_last_cuda_error": (ctypes.c_char_p, []),
    "sda_abi_version": (_i32, []),
    "sda_decode_workspace_size": (_i32, [_i32, _i32, _i32, _i64, ctypes.POINTER(ctypes.c_size_t)]),
    "sda_decode": (_i32, [_vp, _vp, _i64, _vp, _i64, _vp, _vp, _f32, _i32, _i32, _i32, _vp, _vp,
                          ctypes.c_size_t, _vp]),
    "sda_decode_fp8_workspace_size": (_i32, [_i32, _i32, _i32, _i64,
                                             ctypes.POINTER(ctypes.c_size_t)]),
    "sda_decode_fp8": (_i32, [_vp, _vp, _vp, _i64, _vp, _i64, _vp, _vp, _f32, _i32, _i32, _i32, _vp,
                              _vp, ctypes.c_size_t, _vp]),
    "sda_decode_noalloc": (_i32, [_vp, _vp, _i64, _vp, _i64, _vp, _vp, _f32, _i32, _i32, _i32, _vp,
                                  _vp]),
    "sda_decode_error_flag": (_i32, [_vp, _vp, _vp]),
    "sda_decode_kernel": (_i32, [_i32, _i32, _vp]),
    "sda_set_timing_events": (_i32, [_vp, _vp]),
    "sda_debug_wait_fault": (_i32, [_i32, ctypes.c_uint64]),
    "sda_build_indices": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _i64, _i64,
                                 _vp, _i64, _vp, _vp, _vp]),
    "sda_validate_indices": (_i32, [_vp, _i64, _vp, _i32, _i64, _vp, _vp]),
    "sda_build_decode_host_workspace_size": (_i32, [_i32, _i32, _i32, _i64, _i64, _i32,
                                                    ctypes.POINTER(ctypes.c_size_t)]),
    "sda_build_decode_host": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i64, _i64, _vp,
                                     _vp, _vp, _i64, _vp, _f32, _i32, _i32, _i32, _vp, _vp, _vp,
                                     ctypes.c_size_t, _vp]),
    "sda_build_decode": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i64, _vp, _i64, _vp,
                                _vp, _vp, _vp, _vp, _i64, _vp, _f32, _i32, _i32, _i32, _vp, _vp,
                                ctypes.c_size_t, _vp]),
    "sda_topk_slots": (_i32, [_vp, _i64, _vp, _vp, _i64, _i32, _i32, _i32, _vp, _vp, _vp, _i64, _vp,
                              _vp]),
    "sda_qk_norm_rope_swa_store": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32,
                                          _i32, _i32, _f32, _i32, _i64, _i64, _vp, _vp, _vp, _vp]),
    "sda_qk_norm_rope_swa_store_fp8": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32,
                                              _i32, _i32, _i32, _f32, _i32, _i64, _i64, _vp, _vp,
                                              _vp, _vp, _vp]),
}


class SdaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        lib = _lib
        msg = lib.sda_strerror(code).decode() if lib is not None else STATUS_NAMES.get(code, str(code))
        cuda = lib.sda_last_cuda_error().decode() if (lib is not None and code == 3) else ""
        super().__init__(f"{what}: {msg}" + (f" [{cuda}]" if cuda else ""))


def load():
    """Load libsda.so (built by ``python -m sink_sda_decode_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libsda.so not found at {LIB_PATH}: build it first "
                "(python -m sink_sda_decode_gb300.build); there is no fallback path")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def check(code: int, what: str):
    if code != SDA_OK:
        raise SdaError(code, what)
