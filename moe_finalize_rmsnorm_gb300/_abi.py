"""ctypes declarations of include/moe_finalize.h (libmoe_finalize.so).

Loading fails loudly when the library is missing: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

MF_OK = 0
STATUS_NAMES = {
    0: "MF_OK", 1: "MF_ERR_NULL", 2: "MF_ERR_SHAPE", 3: "MF_ERR_ALIGN", 4: "MF_ERR_DTYPE",
    5: "MF_ERR_UNSUPPORTED", 6: "MF_ERR_CUDA", 7: "MF_ERR_DEVICE_TIMEOUT", 8: "MF_ERR_INVALID",
}
MF_DTYPE_BF16, MF_DTYPE_FP32, MF_DTYPE_PACKED_TOPK = 0, 1, 2
VARIANTS = {"auto": 0, "token_cta": 1, "bulk": 2, "cluster": 3}
VARIANT_NAMES = {v: k for k, v in VARIANTS.items()}

# Every exported symbol with (restype, argtypes).
_vp, _i64, _i32, _f32, _int, _u64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                     ctypes.c_float, ctypes.c_int, ctypes.c_uint64)
_TP_ARGS = [_vp, _i64, _i64, _vp, _int, _vp, _vp, _vp, _i64, _i32, _i32, _f32, _f32, _int]
_BEAM_ARGS = [_vp, _i64, _vp, _i64, _vp, _i64, _i32, _i32, _f32, _vp, _f32, _int]
SIGNATURES = {
    "moe_finalize_rmsnorm": (_int, _TP_ARGS + [_vp]),
    "moe_finalize_rmsnorm_variant": (_int, _TP_ARGS + [_int, _vp]),
    "beam_moe_finalize": (_int, _BEAM_ARGS + [_vp]),
    "beam_moe_finalize_variant": (_int, _BEAM_ARGS + [_int, _vp]),
    "beam_moe_finalize_norm_residual_norm": (
        _int, [_vp, _i64, _vp, _i64, _vp, _i64, _i32, _i32, _f32, _vp, _f32, _int, _vp, _f32,
               _int, _f32, _f32, _vp, _vp, _vp]),
    "mf_finalize_data_movement": (_int, [_vp, _i64, _i64, _vp, _int, _vp, _vp, _i64, _vp]),
    "mf_select_finalize_variant": (_int, [_i64, _i32, _i32]),
    "mf_select_beam_variant": (_int, [_i64, _i32, _i32]),
    "mf_finalize_kernel_name": (ctypes.c_char_p, [_i64, _i32, _i32, _int]),
    "mf_beam_kernel_name": (ctypes.c_char_p, [_i64, _i32, _i32, _int, _int]),
    "mf_status_string": (ctypes.c_char_p, [_int]),
    "mf_device_status": (_int, [_int]),
    "mf_selftest_wait_timeout": (_int, [_u64, _vp]),
    "mf_version": (_i32, []),
    "mf_set_programmatic_launch": (None, [_int]),
    "mf_get_programmatic_launch": (_int, []),
}

_lock = threading.Lock()
_lib = None


class MoeFinalizeError(RuntimeError):
    """A non-MF_OK status from the library."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        name = STATUS_NAMES.get(self.status, str(status))
        try:
            msg = lib().mf_status_string(self.status).decode()
        except Exception:  # pragma: no cover - message lookup only
            msg = ""
        super().__init__(f"{where}: {name} ({msg})")


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise ImportError(
                    f"{LIB} is missing: build it with `python -m moe_finalize_rmsnorm_gb300.build` "
                    "(the finalize path has no CPU fallback)")
            handle = ctypes.CDLL(LIB)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def check(status: int, where: str) -> None:
    if status != MF_OK:
        raise MoeFinalizeError(status, where)
