"""ctypes binding of libwise.so (the C ABI declared in include/wise.h).

Argument marshalling only: every computation runs in the library's CUDA
kernels. Loading fails loudly when the library is missing and cannot be
built; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

WISE_OK = 0
WISE_ERR_INVALID_ARGUMENT = 1
WISE_ERR_UNSUPPORTED = 2
WISE_ERR_ALIGNMENT = 3
WISE_ERR_WORKSPACE = 4
WISE_ERR_BAD_SUPPORT = 5
WISE_ERR_CUDA = 6
WISE_ERR_DEVICE_TIMEOUT = 7

WISE_BF16 = 0
WISE_F32 = 1
WISE_SUPPORT_SINK = 1
WISE_SUPPORT_DIAG = 2
WISE_CONTROL_MASS_MATCHED = 1
WISE_CONTROL_SIZE_MATCHED = 2

# Every symbol include/wise.h declares.
EXPORTS = (
    "wise_abi_version", "wise_status_str", "wise_attn_discover_workspace", "wise_attn_discover",
    "wise_schedule_units", "wise_support_capacity", "wise_select_workspace", "wise_select_support",
    "wise_attn_sparse", "wise_validate_support", "wise_device_status", "wise_select_support_noalloc",
    "wise_support_retained_mass", "wise_support_jaccard", "wise_select_control", "wise_attn_discover_select",
    "wise_select_finalize", "wise_validate_schedule", "wise_wait_expiry_check", "wise_gather_plan_bytes",
    "wise_gather_plan", "wise_attn_sparse_planned",
)


class WiseError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} (status {status})" if what else status_str(status))


class AttnDesc(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("heads", ctypes.c_int32),
        ("seq_len", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("out_dtype", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32),
    ]


_lock = threading.Lock()
_handle = None

_vp = ctypes.c_void_p
_sz = ctypes.c_size_t
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_u32 = ctypes.c_uint32
_dp = ctypes.POINTER(AttnDesc)

_SIGNATURES = {
    "wise_abi_version": (ctypes.c_int, []),
    "wise_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "wise_attn_discover_workspace": (_sz, [_dp]),
    "wise_attn_discover": (ctypes.c_int, [_dp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "wise_schedule_units": (_i64, [_dp]),
    "wise_support_capacity": (_i64, [_dp]),
    "wise_select_workspace": (_sz, [_dp, _i32]),
    "wise_select_support": (ctypes.c_int, [_dp, _vp, _i32, ctypes.c_double, _u32, _vp, _vp, _i64, _vp, _vp, _vp,
                                           _sz, _vp]),
    "wise_select_support_noalloc": (ctypes.c_int, [_dp, _vp, _i32, ctypes.c_double, _u32, _vp, _vp, _i64, _vp,
                                                   _vp, _vp]),
    "wise_attn_sparse": (ctypes.c_int, [_dp, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp]),
    "wise_validate_support": (ctypes.c_int, [_dp, _vp, _vp, _u32]),
    "wise_select_control": (ctypes.c_int, [_dp, _vp, _i32, _vp, _vp, _i64, _u32, _vp, _vp, _i64, _vp, _vp, _vp,
                                           _sz, _vp]),
    "wise_support_retained_mass": (ctypes.c_int, [_dp, _vp, _vp, _vp, _i64, _vp, _vp, _vp]),
    "wise_support_jaccard": (ctypes.c_int, [_dp, _vp, _vp, _i64, _vp, _vp, _i64, _vp, _vp, _vp, _vp]),
    "wise_attn_discover_select": (ctypes.c_int, [_dp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, ctypes.c_double, _u32,
                                                 _i32, _i32, _vp, _sz, _vp]),
    "wise_select_finalize": (ctypes.c_int, [_dp, _vp, _sz, _vp, _vp, _i64, _vp, _vp, _vp]),
    "wise_validate_schedule": (ctypes.c_int, [_dp, _vp]),
    "wise_gather_plan_bytes": (ctypes.c_size_t, [_dp]),
    "wise_gather_plan": (ctypes.c_int, [_dp, _vp, _vp, _i64, _vp, ctypes.c_size_t, _vp]),
    "wise_attn_sparse_planned": (ctypes.c_int, [_dp, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp]),
    "wise_wait_expiry_check": (ctypes.c_int, [_vp]),
    "wise_device_status": (ctypes.c_int, [_vp]),
}


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libwise.so (building it first if it is missing or stale and nvcc
    is available). Raises if the library cannot be had."""
    global _handle
    with _lock:
        if _handle is not None:
            return _handle
        if build_if_missing:
            try:
                _build.build()
            except RuntimeError:
                if not os.path.exists(_build.LIB_PATH):
                    raise
        if not os.path.exists(_build.LIB_PATH):
            raise RuntimeError(f"{_build.LIB_PATH} is missing: build the CUDA library first")
        lib = ctypes.CDLL(_build.LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _handle = lib
        return lib


def status_str(status: int) -> str:
    return load().wise_status_str(status).decode()


def check(status: int, what: str = "") -> None:
    if status != WISE_OK:
        raise WiseError(status, what)


def make_desc(batch: int, heads: int, seq_len: int, head_dim: int, block: int, scale: float = 0.0,
              out_dtype: int = WISE_BF16, kv_heads: int = 0) -> AttnDesc:
    return AttnDesc(batch, heads, seq_len, head_dim, block, scale, out_dtype, kv_heads)
