"""ctypes view of ``include/fm.h``: structures, status codes and the loaded
library.  Argument marshalling only; no arithmetic happens here."""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfm.so")

FM_OK, FM_ERR_INVALID, FM_ERR_BOUNDS, FM_ERR_UNSUPPORTED, FM_ERR_WORKSPACE, FM_ERR_CUDA, \
    FM_ERR_TIMEOUT = range(7)

STATUS_NAMES = {
    FM_OK: "FM_OK", FM_ERR_INVALID: "FM_ERR_INVALID", FM_ERR_BOUNDS: "FM_ERR_BOUNDS",
    FM_ERR_UNSUPPORTED: "FM_ERR_UNSUPPORTED", FM_ERR_WORKSPACE: "FM_ERR_WORKSPACE",
    FM_ERR_CUDA: "FM_ERR_CUDA", FM_ERR_TIMEOUT: "FM_ERR_TIMEOUT",
}


class FmDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("Hm", ctypes.c_int),
                ("Sq", ctypes.c_int), ("Skv", ctypes.c_int), ("d", ctypes.c_int),
                ("Hkv", ctypes.c_int),
                ("q_stride", ctypes.c_int64 * 3), ("k_stride", ctypes.c_int64 * 3),
                ("v_stride", ctypes.c_int64 * 3), ("o_stride", ctypes.c_int64 * 3)]


class FmWsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "status", "summary", "table", "row_count", "row_list", "col_count", "col_list",
        "fwd_order", "bwd_order", "row_mask", "masks", "pair_info", "pair_list", "delta",
        "lse_log2", "row_order", "total")]


class FMError(RuntimeError):
    """A non-OK status returned by the library."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({status_string(code)})")


_lib = None

P = ctypes.c_void_p
I32P = ctypes.c_void_p

SIGNATURES = {
    "fm_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(FmDesc), ctypes.c_int]),
    "fm_workspace_layout": (ctypes.c_int, [ctypes.POINTER(FmDesc), ctypes.c_int,
                                           ctypes.POINTER(FmWsLayout)]),
    "fm_plan": (ctypes.c_int, [ctypes.POINTER(FmDesc), I32P, I32P, I32P, I32P, P, ctypes.c_size_t,
                               ctypes.c_int, P]),
    "fm_fwd": (ctypes.c_int, [ctypes.POINTER(FmDesc), P, P, P, I32P, I32P, I32P, I32P,
                              ctypes.c_float, P, P, P, ctypes.c_size_t, P]),
    "fm_bwd": (ctypes.c_int, [ctypes.POINTER(FmDesc), P, P, P, P, P, P, I32P, I32P, I32P, I32P,
                              ctypes.c_float, P, P, P, P, ctypes.c_size_t, P]),
    "fm_fwd_planned": (ctypes.c_int, [ctypes.POINTER(FmDesc), P, P, P, I32P, I32P, I32P, I32P,
                                      ctypes.c_float, P, P, P, ctypes.c_size_t, P]),
    "fm_bwd_planned": (ctypes.c_int, [ctypes.POINTER(FmDesc), P, P, P, P, P, P, I32P, I32P, I32P,
                                      I32P, ctypes.c_float, P, P, P, P, ctypes.c_size_t, P]),
    "fm_fwd_static": (ctypes.c_int, [ctypes.POINTER(FmDesc), P, P, P, I32P, I32P, I32P, I32P,
                                     ctypes.c_float, P, P, P]),
    "fm_quantize_fp8": (ctypes.c_int, [ctypes.POINTER(FmDesc), P, P, P, P, P, P, P, P, P, P, P]),
    "fm_fwd_fp8": (ctypes.c_int, [ctypes.POINTER(FmDesc), P, P, P, P, P, P, P, I32P, I32P, I32P,
                                  I32P, ctypes.c_float, P, P, P, ctypes.c_size_t, P]),
    "fm_varlen_bounds": (ctypes.c_int, [I32P, ctypes.c_int, ctypes.c_int, ctypes.c_int, I32P, P,
                                        P]),
    "fm_localize": (ctypes.c_int, [I32P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P,
                                   ctypes.c_int, I32P, P]),
    "fm_device_status": (ctypes.c_int, [P, P]),
    "fm_test_hooks": (ctypes.c_int, [ctypes.c_uint64, ctypes.c_int]),
    "fm_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fm_version": (ctypes.c_int, []),
    "fm_profile_enable": (ctypes.c_int, [ctypes.c_int]),
    "fm_profile_read": (ctypes.c_int, [P, P, ctypes.c_int]),
    "fm_kernel_name": (ctypes.c_char_p, [ctypes.c_int]),
    "fm_measure_exp2_rate": (ctypes.c_int, [P, P]),
}

KERNEL_IDS = 11


def lib():
    """The loaded ``libfm.so``.  Raises if it has not been built: there is no
    other implementation to fall back to."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -m masked_attention_bound_gb300.build, or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(code: int) -> str:
    try:
        return lib().fm_status_string(code).decode()
    except Exception:  # the library may be missing while formatting an error
        return STATUS_NAMES.get(code, str(code))


def check(code: int, where: str):
    if code != FM_OK:
        raise FMError(code, where)
