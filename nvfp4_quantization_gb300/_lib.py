"""ctypes loader for libepq.so (the C ABI declared in include/epq.h).

The library is built in-tree by ``nvfp4_quantization_gb300.build``; if it is
missing it is built on first use, and if that is impossible the import fails
loudly -- there is no fallback implementation of any kernel.
"""
from __future__ import annotations

import ctypes
import threading

from . import build as _build

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int
_U64 = ctypes.c_uint64

EP_OK = 0
EP_ROUND_RNE = 0
EP_ROUND_SR = 1
EP_DEV_ERR_BAD_EXPERT = 1
EP_DEV_ERR_DUP_EXPERT = 2
EP_DEV_ERR_TIMEOUT = 4
EP_DEV_ERR_CAPACITY = 8
EP_ROUTE_STATIC_SCRATCH_BYTES = 262144   # mirrors the macro in include/epq.h

# every symbol include/epq.h declares
SYMBOLS = ("ep_nvfp4_row_bytes", "ep_rows_capacity", "ep_route_workspace_bytes", "ep_route_plan",
           "ep_route_plan_noalloc", "ep_nvfp4_pack", "ep_nvfp4_dispatch", "ep_nvfp4_unpack", "ep_nvfp4_direct_receive",
           "ep_nvfp4_direct_receive_swizzled", "ep_nvfp4_colwise_rht_bf16", "ep_mxfp8_pack",
           "ep_mxfp8_colwise", "ep_status_string")


class EpGrouped(ctypes.Structure):
    """Mirror of ep_nvfp4_grouped."""
    _fields_ = [("rw_codes", _P), ("rw_scales", _P), ("rw_row_scale", _P), ("cw_codes", _P),
                ("cw_scales", _P), ("amax_row", _P), ("amax_col", _P), ("cw_scale_enc", _P)]


class EpError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


_lock = threading.Lock()
_lib = None


def _declare(L):
    L.ep_nvfp4_row_bytes.argtypes = [_I64]; L.ep_nvfp4_row_bytes.restype = ctypes.c_size_t
    L.ep_rows_capacity.argtypes = [_I64, _I32, _I32, _I32]; L.ep_rows_capacity.restype = _I64
    L.ep_route_workspace_bytes.argtypes = [_I64, _I32, _I32]; L.ep_route_workspace_bytes.restype = ctypes.c_size_t
    L.ep_route_plan.argtypes = [_P, _I64, _I32, _I32, _I32, _I64, _P, _P, _P, _P, ctypes.c_size_t, _P, _P]
    L.ep_route_plan.restype = _I32
    L.ep_route_plan_noalloc.argtypes = [_P, _I64, _I32, _I32, _I32, _I64, _P, _P, _P, _P, _P]
    L.ep_route_plan_noalloc.restype = _I32
    L.ep_nvfp4_pack.argtypes = [_P, _I64, _I64, _P, _I32, _P, _P, _I32, _P, _I64, _P, _I32, _U64, _P, _P]
    L.ep_nvfp4_pack.restype = _I32
    L.ep_nvfp4_dispatch.argtypes = [_P, _P, _I64, _I64, _I32, _I32, _I32, _I64, _P, _P, _P, _P, ctypes.c_size_t, _P,
                                    _P, _I32, _U64, _P, _P]
    L.ep_nvfp4_dispatch.restype = _I32
    L.ep_nvfp4_unpack.argtypes = [_P, _I64, _I64, _P, _I32, _P, _P, _P]
    L.ep_nvfp4_unpack.restype = _I32
    L.ep_nvfp4_direct_receive.argtypes = [_P, _I64, _I64, _P, _I32, _P, ctypes.POINTER(EpGrouped), _I32, _U64,
                                          ctypes.c_uint16, _P, _P]
    L.ep_nvfp4_direct_receive.restype = _I32
    L.ep_nvfp4_direct_receive_swizzled.argtypes = L.ep_nvfp4_direct_receive.argtypes
    L.ep_nvfp4_direct_receive_swizzled.restype = _I32
    L.ep_nvfp4_colwise_rht_bf16.argtypes = [_P, _I64, _I64, _P, _I32, _P, _P, _P, _P, _P, _P, _I32, _U64,
                                            ctypes.c_uint16, _P, _P]
    L.ep_nvfp4_colwise_rht_bf16.restype = _I32
    L.ep_mxfp8_colwise.argtypes = [_P, _I64, _I64, _P, _I32, _P, _P, _P]
    L.ep_mxfp8_colwise.restype = _I32
    L.ep_mxfp8_pack.argtypes = [_P, _I64, _I64, _P, _I32, _P, _P, _I32, _P, _I64, _P, _P]
    L.ep_mxfp8_pack.restype = _I32
    L.ep_status_string.argtypes = [_I32]; L.ep_status_string.restype = ctypes.c_char_p


def lib() -> ctypes.CDLL:
    """The loaded libepq.so (built first if needed)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(str(path))
            _declare(L)
            _lib = L
    return _lib


def library_path() -> str:
    return str(_build.LIB)


def status_string(status: int) -> str:
    return lib().ep_status_string(int(status)).decode()


def check(fn: str, status: int) -> None:
    if status != EP_OK:
        raise EpError(fn, status)
