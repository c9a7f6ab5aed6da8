"""ctypes binding of libfkl.so (argument marshalling only).

The library is loaded from this package's directory on first use.  There is no
fallback: if libfkl.so is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfkl.so")

_lock = threading.Lock()
_lib = None

c_int, c_i64, c_size, c_float, c_double, c_void_p, c_char_p = (
    ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float, ctypes.c_double,
    ctypes.c_void_p, ctypes.c_char_p)

# name -> (restype, argtypes); mirrors include/fkl.h
SIGNATURES = {
    "fkl_workspace_size": (c_size, [c_i64, c_int, c_i64, c_int, c_int]),
    "fkl_forward": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_i64, c_int, c_i64,
                            c_int, c_float, c_int, c_void_p, c_void_p, c_void_p, c_size, c_void_p]),
    "fkl_backward": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_i64, c_int, c_i64,
                             c_int, c_float, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_void_p, c_size, c_void_p]),
    "fkl_mix_forward": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_i64, c_int,
                                c_i64, c_int, c_float, c_float, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_size, c_void_p]),
    "fkl_mix_backward": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_i64, c_int,
                                 c_i64, c_int, c_float, c_float, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                 c_void_p, c_void_p, c_size, c_void_p]),
    "fkl_forward_backward": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_i64, c_int,
                                     c_i64, c_int, c_float, c_int, c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_size, c_void_p]),
    "fkl_forward_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_i64, c_int,
                                    c_i64, c_int, c_float, c_int, c_void_p, c_void_p, c_void_p,
                                    c_void_p]),
    "fkl_topk_workspace_size": (c_size, [c_i64, c_int, c_i64, c_int, c_int]),
    "fkl_teacher_topk": (c_int, [c_void_p, c_void_p, c_i64, c_int, c_i64, c_int, c_int, c_void_p, c_void_p,
                                 c_void_p, c_size, c_void_p]),
    "fkl_scale_grads": (c_int, [c_void_p, c_void_p, c_i64, c_int, c_i64, c_void_p, c_void_p]),
    "fkl_get_status": (c_int, [c_void_p, c_void_p]),
    "fkl_status_string": (c_char_p, [c_int]),
    "fkl_last_error": (c_char_p, []),
    "fkl_profile_enable": (None, [c_int]),
    "fkl_profile_reset": (None, []),
    "fkl_profile_read": (c_int, [ctypes.POINTER(c_double), ctypes.POINTER(c_i64),
                                 ctypes.POINTER(c_double), c_int]),
    "fkl_kernel_name": (c_char_p, [c_int]),
    "fkl_launch_count": (c_i64, []),
    "fkl_selftest_wait_timeout": (c_int, [c_void_p, c_i64, c_void_p]),
    "fkl_selftest_gemm": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int,
                                  c_int, c_void_p, c_void_p]),
}


def lib():
    """The loaded library (raises OSError if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise OSError(f"{LIB_PATH} is missing: build it with "
                              "`python -m lm_head_kl_fkl_b300.build`")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib
