"""ctypes declarations of the C ABI in include/attn_fwd.h.

Loading builds the in-tree library first if it is missing or older than its
sources (the CUDA sources are the product; there is no other code path).  If
the library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import threading

from . import build as _build


class attn_strides(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("head", ctypes.c_int64), ("row", ctypes.c_int64)]


class attn_opts(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_float), ("causal", ctypes.c_int), ("softcap", ctypes.c_float),
                ("sink", ctypes.c_void_p), ("use_window", ctypes.c_int),
                ("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
                ("top_left", ctypes.c_int), ("alibi_slopes", ctypes.c_void_p),
                ("alibi_stride", ctypes.c_int), ("bias", ctypes.c_void_p),
                ("bias_strides", attn_strides), ("scale_p", ctypes.c_float),
                ("scale_o", ctypes.c_float)]


STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_CUDA",
          4: "ATTN_ERR_TIMEOUT"}
ATTN_F16, ATTN_BF16, ATTN_E4M3 = 0, 1, 2

EXPORTS = ("attn_fwd", "attn_fwd_varlen", "attn_fwd_paged", "attn_splitkv_combine",
           "attn_paged_workspace_bytes", "attn_paged_auto_splits", "attn_status_string",
           "attn_last_kernel_name", "attn_device_error", "attn_selftest_timeout",
           "attn_fwd_paged_noalloc", "attn_paged_window_pages", "attn_dense_schedule")
NOALLOC_SCRATCH_BYTES = 16 << 20

_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int


def _declare(lib):
    S = attn_strides
    O = ctypes.POINTER(attn_opts)
    lib.attn_fwd.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, S, S, S, S, O, _P]
    lib.attn_fwd_varlen.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                    S, S, S, S, O, _P]
    lib.attn_fwd_paged.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                   _I, _I, _P, _P, O, _P]
    lib.attn_fwd_paged_noalloc.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                           _I, _I, _I, _I, O, _P]
    lib.attn_splitkv_combine.argtypes = [_P, _P, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P]
    lib.attn_paged_workspace_bytes.argtypes = [_I, _I, _I, _I, _I]
    lib.attn_paged_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_paged_auto_splits.argtypes = [_I, _I, _I]
    lib.attn_paged_auto_splits.restype = _I
    lib.attn_paged_window_pages.argtypes = [_I, _I, _I, O]
    lib.attn_paged_window_pages.restype = _I
    IP = ctypes.POINTER(ctypes.c_int32)
    lib.attn_dense_schedule.argtypes = [_I, _I, _I, _I, _I, O, _I, IP, IP]
    lib.attn_dense_schedule.restype = _I
    lib.attn_status_string.argtypes = [_I]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_last_kernel_name.argtypes = []
    lib.attn_last_kernel_name.restype = ctypes.c_char_p
    lib.attn_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint)]
    lib.attn_selftest_timeout.argtypes = [ctypes.c_uint64, _P]
    for name in ("attn_fwd", "attn_fwd_varlen", "attn_fwd_paged", "attn_splitkv_combine",
                 "attn_device_error", "attn_selftest_timeout", "attn_fwd_paged_noalloc"):
        getattr(lib, name).restype = _I


def load(build: bool = True) -> ctypes.CDLL:
    """Load libattn_fwd.so (building it first when ``build`` and it is stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build else _build.LIB
            lib = ctypes.CDLL(path)
            _declare(lib)
            _lib = lib
        return _lib


def lib_path() -> str:
    return _build.LIB
