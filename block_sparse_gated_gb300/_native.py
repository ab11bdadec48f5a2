"""ctypes binding of libbsfa.so (declared in include/bsfa.h).

Loads the in-tree library on first use and raises if it has not been built:
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbsfa.so")

c_int, c_float, c_void_p, c_size_t = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
c_int64 = ctypes.c_int64


class FwdParams(ctypes.Structure):
    """Mirror of bsfa_fwd_params."""
    _fields_ = [
        ("q", c_void_p), ("k", c_void_p), ("v", c_void_p), ("o", c_void_p),
        ("q_stride", c_int64 * 3), ("k_stride", c_int64 * 3),
        ("v_stride", c_int64 * 3), ("o_stride", c_int64 * 3),
        ("batch", c_int), ("num_heads_q", c_int), ("num_heads_kv", c_int),
        ("seqlen", c_int), ("head_dim", c_int),
        ("cu_seqlens", c_void_p), ("max_seqlen", c_int),
        ("block_q", c_int), ("block_k", c_int),
        ("softmax_scale", c_float), ("mode", c_int),
        ("thresholds", c_void_p), ("thresholds_nq", c_int),
        ("log_lambda", c_float),
        ("kept_bitmap", c_void_p), ("lse", c_void_p), ("block_counts", c_void_p),
        ("workspace", c_void_p), ("workspace_bytes", c_size_t),
        ("dtype", c_int), ("flags", ctypes.c_uint),
        ("block_table", c_void_p), ("block_table_stride", c_int),
        ("page_size", c_int), ("num_pages", c_int),
    ]


# bsfa_dtype
DTYPE_BF16, DTYPE_F16 = 0, 1
# bsfa_flag
FLAG_V_ALWAYS = 1
FLAG_MEAN_CORRECTION = 2
FLAG_PIPELINED = 4


# Every exported symbol and its C signature: (name, restype, argtypes).
SIGNATURES = [
    ("bsfa_version", c_int, []),
    ("bsfa_status_string", ctypes.c_char_p, [c_int]),
    ("bsfa_prefill_workspace_size", c_size_t, [ctypes.POINTER(FwdParams)]),
    ("bsfa_bitmap_words_per_row", c_int, [ctypes.POINTER(FwdParams), ctypes.POINTER(c_int)]),
    ("bsfa_prefill_fwd", c_int, [ctypes.POINTER(FwdParams), c_void_p]),
    ("bsfa_calibrate_workspace_size", c_size_t, [c_int, c_int, c_int, c_int]),
    ("bsfa_calibrate", c_int, [
        ctypes.POINTER(c_void_p), ctypes.POINTER(c_void_p), c_int, c_int, c_int, c_int, c_int,
        c_int, ctypes.POINTER(c_int64), ctypes.POINTER(c_int64), c_int, c_int, c_float,
        ctypes.POINTER(c_int), c_int, c_void_p, c_void_p, c_size_t, c_void_p]),
    ("bsfa_device_error", c_int, [c_void_p, ctypes.POINTER(ctypes.c_uint)]),
    ("bsfa_prefill_fwd_noalloc", c_int, [ctypes.POINTER(FwdParams), c_void_p]),
    ("bsfa_selftest_wait_guard", c_int, [ctypes.c_uint, c_void_p]),
]

_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built: run `python -m block_sparse_gated_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib
