"""ctypes loader of libsdpa.so with the C signatures of include/sdpa.h.

Argument marshalling only. The library is required: there is no fallback, and
every function raises when the shared object has not been built.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsdpa.so")

SDPA_OK = 0
SDPA_ERR_INVALID_ARG = 1
SDPA_ERR_UNSUPPORTED = 2
SDPA_ERR_MISALIGNED = 3
SDPA_ERR_WORKSPACE = 4
SDPA_ERR_CUDA = 5
SDPA_ERR_DEVICE_TIMEOUT = 6
SDPA_BWD_PREPROCESS = 1
SDPA_BWD_DKDV = 2
SDPA_BWD_DQ = 4
SDPA_BWD_ALL = 7
SDPA_BWD_DETERMINISTIC = 8
SDPA_BF16 = 0
SDPA_FP16 = 1

# name -> (restype, argtypes), in the order of include/sdpa.h
_i64, _f32, _int, _u64, _ptr, _sz = (ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_uint64,
                                     ctypes.c_void_p, ctypes.c_size_t)
SIGNATURES = {
    "sdpa_fwd": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _f32, _int, _f32, _u64, _u64, _int,
                        _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr]),
    "sdpa_bwd_workspace_size": (_sz, [_i64, _i64, _i64, _i64, _i64, _i64]),
    "sdpa_bwd_workspace_size_ex": (_sz, [_i64, _i64, _i64, _i64, _i64, _i64, _i64, _int]),
    "sdpa_bwd_workspace_size_gqa": (_sz, [_i64, _i64, _i64, _i64, _i64, _i64, _i64]),
    "sdpa_bwd": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _f32, _int, _f32, _u64, _u64, _int,
                        _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr,
                        _sz, _ptr]),
    "sdpa_bwd_phases": (_int, [_int, _i64, _i64, _i64, _i64, _i64, _i64, _f32, _int, _f32, _u64,
                               _u64, _int, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr,
                               _ptr, _ptr, _ptr, _sz, _ptr]),
    "sdpa_fwd_gqa": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _i64, _f32, _int, _f32, _u64, _u64,
                            _int, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr]),
    "sdpa_bwd_gqa": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _i64, _f32, _int, _f32, _u64, _u64,
                            _int, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr,
                            _ptr, _sz, _ptr]),
    "sdpa_bwd_phases_gqa": (_int, [_int, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _f32, _int, _f32,
                                   _u64, _u64, _int, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr,
                                   _ptr, _ptr, _ptr, _ptr, _sz, _ptr]),
    "sdpa_bwd_varlen_workspace_size": (_sz, [_i64, _i64, _i64]),
    "sdpa_bwd_varlen_workspace_size_ex": (_sz, [_i64, _i64, _i64, _i64, _int]),
    "sdpa_fwd_varlen": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _f32, _int, _f32,
                               _u64, _u64, _int, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr]),
    "sdpa_bwd_varlen": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _f32, _int, _f32,
                               _u64, _u64, _int, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr,
                               _ptr, _ptr, _ptr, _sz, _ptr]),
    "sdpa_bwd_phases_varlen": (_int, [_int, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _f32,
                                      _int, _f32, _u64, _u64, _int, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr,
                                      _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _sz, _ptr]),
    "sdpa_fwd_ex": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _i64, _f32, _i64, _i64, _int, _ptr, _i64, _ptr, _ptr, _f32, _u64,
                               _u64, _int, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr]),
    "sdpa_bwd_ex": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _i64, _f32, _i64, _i64, _int, _ptr, _i64, _ptr, _f32, _u64,
                               _u64, _int, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _sz,
                               _ptr]),
    "sdpa_bwd_phases_ex": (_int, [_int, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _f32, _i64, _i64, _int, _ptr, _i64, _ptr, _f32,
                                      _u64, _u64, _int, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr,
                                      _sz, _ptr]),
    "sdpa_fwd_varlen_ex": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _f32, _i64, _i64, _int, _ptr, _i64, _ptr,
                                      _ptr, _f32, _u64, _u64, _int, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr]),
    "sdpa_bwd_varlen_ex": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _f32, _i64, _i64, _int, _ptr, _i64, _ptr,
                                      _f32, _u64, _u64, _int, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr,
                                      _ptr, _sz, _ptr]),
    "sdpa_bwd_phases_varlen_ex": (_int, [_int, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _i64, _f32, _i64, _i64, _int, _ptr,
                                             _i64, _ptr, _f32, _u64, _u64, _int, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr,
                                             _ptr, _ptr, _sz, _ptr]),
    "sdpa_bwd_noalloc": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _f32, _int, _f32, _u64, _u64,
                                _int, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr, _ptr,
                                _ptr, _ptr]),
    "sdpa_dropout_mask": (_int, [_i64, _i64, _i64, _i64, _f32, _u64, _u64, _ptr, _ptr]),
    "sdpa_device_error": (_int, [ctypes.POINTER(ctypes.c_uint32), _int]),
    "sdpa_debug_fault": (_int, [_int, ctypes.c_uint64]),
    "sdpa_tile_ranges": (_i64, [_int, _i64, _i64, _i64, _i64, _int, _int, _int, _ptr, _i64]),
    "sdpa_last_error": (ctypes.c_char_p, []),
    "sdpa_status_string": (ctypes.c_char_p, [_int]),
    "sdpa_version": (_int, []),
}

_lib = None


class SdpaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


def lib() -> ctypes.CDLL:
    """The loaded library (built by scaled_dot_product_06_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().sdpa_status_string(int(status)).decode()


def check(status: int, what: str) -> None:
    if status != SDPA_OK:
        detail = lib().sdpa_last_error().decode()
        raise SdpaError(status, f"{what} ({detail})" if detail else what)
