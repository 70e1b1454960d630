"""ctypes view of libmgg.so (declarations mirror include/mgg.h and include/mgg_testing.h)."""
from __future__ import annotations

import ctypes
import os
import threading
from ctypes import c_char_p, c_int, c_int32, c_int64, c_size_t, c_uint32, c_uint64, c_void_p

# MGG_LIB_VARIANT=checked loads the bounds-checked debugging build (build.py --checked) instead.
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "libmgg_checked.so" if os.environ.get("MGG_LIB_VARIANT") == "checked" else "libmgg.so")

MGG_OK = 0
MGG_ERR_VALUE = 1
MGG_ERR_UNSUPPORTED = 2
MGG_ERR_RUNTIME = 3
MGG_ERR_ARCH = 4
MGG_ERR_DEVICE_OFFSETS = 5
MGG_ERR_DEVICE_POINTER = 6
MGG_ERR_DEVICE_TIMEOUT = 7
MGG_ERR_DEVICE_BOUNDS = 8

DTYPES = {"bf16": 0, "fp16": 1, "fp32": 2}
ACTS = {"dswiglu": 0, "dgeglu": 1, "dsituglu": 2}
FILTERS = {"value": 0, "indicator": 1}
MAJORS = {"k": 0, "mn": 1, "m": 1, "n": 1}
SCHEDS = {"static": 0, "dynamic": 1}
CTA_MODES = {"auto": 0, "single": 1, "pair": 2}
ORDERS = {"tensor2d": 0, "tensor_ragged": 1}


class DgluBwdArgs(ctypes.Structure):
    _fields_ = [
        ("M", c_int64), ("K", c_int64), ("N", c_int64), ("L", c_int64),
        ("a", c_void_p), ("b", c_void_p), ("b_ptrs", c_void_p), ("c", c_void_p),
        ("padded_offsets", c_void_p), ("alpha", c_void_p), ("beta", c_void_p), ("prob", c_void_p),
        ("dprob", c_void_p), ("d_row", c_void_p), ("dbias", c_void_p), ("d_col", c_void_p), ("amax", c_void_p),
        ("workspace", c_void_p), ("tile_log", c_void_p),
        ("workspace_bytes", c_int64), ("tile_log_capacity", c_int64),
        ("b_major", c_int32), ("c_dtype", c_int32), ("d_dtype", c_int32), ("act", c_int32),
        ("geglu_filter", c_int32), ("gate_first", c_int32), ("sched", c_int32), ("cta_mode", c_int32),
        ("situ_beta1", ctypes.c_float), ("situ_beta2", ctypes.c_float),
    ]


class DsreluBwdArgs(ctypes.Structure):
    _fields_ = [
        ("M", c_int64), ("K", c_int64), ("N", c_int64), ("L", c_int64),
        ("a", c_void_p), ("b", c_void_p), ("b_ptrs", c_void_p), ("c", c_void_p),
        ("padded_offsets", c_void_p), ("alpha", c_void_p), ("prob", c_void_p),
        ("dprob", c_void_p), ("d_row", c_void_p), ("d_col", c_void_p), ("amax", c_void_p),
        ("workspace", c_void_p), ("tile_log", c_void_p),
        ("workspace_bytes", c_int64), ("tile_log_capacity", c_int64),
        ("b_major", c_int32), ("c_dtype", c_int32), ("d_dtype", c_int32), ("sched", c_int32),
        ("cta_mode", c_int32), ("reserved", c_int32),
    ]


class WgradArgs(ctypes.Structure):
    _fields_ = [
        ("hidden", c_int64), ("inter", c_int64), ("L", c_int64), ("tokens_sum", c_int64),
        ("a", c_void_p), ("b", c_void_p), ("offsets", c_void_p), ("out", c_void_p), ("out_ptrs", c_void_p),
        ("workspace", c_void_p), ("tile_log", c_void_p),
        ("workspace_bytes", c_int64), ("tile_log_capacity", c_int64),
        ("a_major", c_int32), ("b_major", c_int32), ("input_order", c_int32), ("out_dtype", c_int32),
        ("accumulate", c_int32), ("sched", c_int32), ("cta_mode", c_int32), ("reserved1", c_int32),
    ]


# (name, restype, argtypes) of every exported function declared in include/*.h
SIGNATURES = [
    ("mgg_abi_version", c_int, []),
    ("mgg_sizeof_dglu_bwd_args", c_size_t, []),
    ("mgg_sizeof_dsrelu_bwd_args", c_size_t, []),
    ("mgg_sizeof_wgrad_args", c_size_t, []),
    ("mgg_args_field_offsets", c_int, [c_int, ctypes.POINTER(c_size_t), c_int]),
    ("mgg_last_error", c_char_p, []),
    ("mgg_status_string", c_char_p, [c_int]),
    ("mgg_dglu_bwd_workspace_size", c_size_t, [c_int64, c_int64]),
    ("mgg_dsrelu_bwd_workspace_size", c_size_t, [c_int64]),
    ("mgg_wgrad_workspace_size", c_size_t, [c_int64]),
    ("mgg_dglu_bwd_num_tiles", c_int64, [c_int64, c_int64]),
    ("mgg_wgrad_num_tiles", c_int64, [c_int64, c_int64, c_int64]),
    ("mgg_dglu_bwd_tile_shape", None, [ctypes.POINTER(c_int32), ctypes.POINTER(c_int32)]),
    ("mgg_wgrad_tile_shape", None, [c_int64, ctypes.POINTER(c_int32), ctypes.POINTER(c_int32)]),
    ("mgg_dglu_bwd", c_int, [ctypes.POINTER(DgluBwdArgs), c_void_p]),
    ("mgg_dsrelu_bwd", c_int, [ctypes.POINTER(DsreluBwdArgs), c_void_p]),
    ("mgg_wgrad", c_int, [ctypes.POINTER(WgradArgs), c_void_p]),
    ("mgg_wgrad_noalloc", c_int, [ctypes.POINTER(WgradArgs), c_void_p]),
    ("mgg_read_device_status", c_int, [c_void_p, c_void_p]),
    ("mgg_test_encode_tmap_2d", c_int, [c_void_p, c_void_p, c_uint64, c_uint64, c_uint64, c_uint32, c_uint32]),
    ("mgg_test_tmap_replace", c_int, [c_void_p, c_void_p, c_void_p, c_uint32, c_uint64, c_int, c_void_p]),
    ("mgg_test_wait_timeout", c_int, [c_void_p, c_int64, c_int32, c_int32, c_void_p]),
    ("mgg_test_build_flags", c_int, []),
    ("mgg_test_bounds_check", c_int, [c_void_p, c_int64, c_int64, c_void_p]),
]

_lib = None
_lock = threading.Lock()


def load() -> ctypes.CDLL:
    """Loads libmgg.so (built in-tree by ``build.py``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with `python -m moe_grouped_gemm_persistent_gb300.build` "
                    "(there is no fallback implementation)")
            lib = ctypes.CDLL(LIB_PATH)
            for name, res, args in SIGNATURES:
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


class MggError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        name = load().mgg_status_string(status).decode()
        super().__init__(f"{name}: {message}")


def check(status: int):
    if status != MGG_OK:
        raise MggError(status, load().mgg_last_error().decode())
