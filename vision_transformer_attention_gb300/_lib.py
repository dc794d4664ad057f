"""ctypes loader for libvta_gb300.so (the C ABI of include/rpe_attn.h).

Loading fails loudly when the library has not been built: there is no CPU
or pure-PyTorch stand-in for any entry point.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libvta_gb300.so")

RPE_OK = 0
RPE_ERR_INVALID_ARG = 1
RPE_ERR_UNSUPPORTED = 2
RPE_ERR_CUDA = 3
RPE_ERR_TIMEOUT = 4
RPE_MAP_PRODUCT = 0
RPE_MAP_EUCLIDEAN = 1
RPE_MAP_CROSS = 2
RPE_MAP_CLIP_PRODUCT = 3
RPE_TERM_K, RPE_TERM_Q, RPE_TERM_V = 1, 2, 4
RPE_TABLES_CROSS = 8
RPE_TABLES_PER_HEAD = 16
RPE_CLS_TOKEN = 32
RPE_DTYPE_BF16, RPE_DTYPE_F32 = 0, 1

# name -> (restype, argtypes) for every symbol the header declares
_i, _u, _d, _p, _u64 = ctypes.c_int, ctypes.c_uint, ctypes.c_double, ctypes.c_void_p, ctypes.c_uint64
SIGNATURES = {
    "rpe_build_bucket_ids": (_i, [_i, _i, _i, _d, _d, _d, _p, _p, ctypes.POINTER(_i), _p]),
    "rpe_attn_fwd": (_i, [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _u, _i, _p, _p]),
    "swin_window_attn_fwd": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _i, _p, _p]),
    "swin_window_attn_fwd_noalloc": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _p, _p]),
    "swin_noalloc_status": (_i, [ctypes.POINTER(_u), _i]),
    "swin_noalloc_status_word": (_i, [ctypes.POINTER(_p)]),
    "swin_window_attn_fwd_fmap": (_i, [_p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _p, _p]),
    "rpe_attn_bias_fwd": (_i, [_p, _p, _p, _p, _i, _p, _i, ctypes.c_uint, _i, _i, _i, _i, _i, _i,
                               _p, _p]),
    "rpe_device_status": (_i, [ctypes.POINTER(_u), _i]),
    "rpe_wait_probe": (_i, [_u64, _p]),
    "rpe_status_string": (ctypes.c_char_p, [_i]),
    "rpe_release_stream": (_i, [_p]),
    "rpe_shutdown": (_i, []),
}

_lib = None


class RpeError(RuntimeError):
    def __init__(self, fn, status):
        msg = lib().rpe_status_string(status).decode()
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


def lib():
    """The loaded library; raises if it was never built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m vision_transformer_attention_gb300.build` (no CPU fallback exists)")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def check(fn, status):
    if status != RPE_OK:
        raise RpeError(fn, status)
