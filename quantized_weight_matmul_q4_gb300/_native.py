"""ctypes loader for libkq.so (the C ABI declared in include/kq.h).

The library is built in-tree by ``build.build()``. There is no fallback: if the
shared library is missing or does not load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

from .build import LIB_PATH, INCLUDE

KQ_OK = 0
KQ_ERR_NULL = 1
KQ_ERR_SHAPE = 2
KQ_ERR_ALIGN = 3
KQ_ERR_TYPE = 4
KQ_ERR_WORKSPACE = 5
KQ_ERR_CUDA = 6
KQ_ERR_DEVICE = 7

KQ_Q4_K = 1
KQ_Q6_K = 2
KQ_TQ4_1S = 3
KQ_Q5_K = 4
KQ_OP_MATVEC = 1
KQ_OP_GEMM = 2
KQ_OP_MOE = 3

KQ_DEVERR_NONE = 0
KQ_DEVERR_WAIT_TIMEOUT = 1
KQ_DEVERR_EXPERT_ID = 2

KQ_GEMM_STATIC_WS_BYTES = 32 << 20

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t

SIGNATURES = {
    "kq_quantize_q8_1": (ctypes.c_int, [_vp, _vp, _i64, _i64, _vp]),
    "kq_matvec": (ctypes.c_int, [ctypes.c_int, _vp, _vp, _vp, _i64, _i64, _vp]),
    "kq_matvec_prefetch": (ctypes.c_int, [ctypes.c_int, _vp, _vp, _vp, _i64, _i64, _vp, ctypes.c_size_t, _vp]),
    "kq_matvec_swiglu": (ctypes.c_int, [ctypes.c_int, _vp, _vp, _vp, _vp, _i64, _i64, _vp]),
    "kq_matvec_rmsnorm": (ctypes.c_int, [ctypes.c_int, _vp, _vp, _vp, ctypes.c_float, _vp, _i64, _i64, _vp]),
    "kq_moe_combine": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, _i32, _vp]),
    "kq_gemm": (ctypes.c_int, [ctypes.c_int, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _sz, _vp]),
    "kq_gemm_noalloc": (ctypes.c_int, [ctypes.c_int, _vp, _vp, _vp, _i64, _i64, _i64, _vp]),
    "kq_moe_grouped_gemm": (ctypes.c_int, [ctypes.c_int, _vp, _i32, _vp, _i32, _vp, _vp, _i64, _i64, _i64,
                                           _vp, _sz, _vp]),
    "kq_workspace_bytes": (_sz, [ctypes.c_int, ctypes.c_int, _i64, _i64, _i64, _i32, _i32]),
    "kq_get_device_error": (ctypes.c_int, [ctypes.POINTER(_i32), _vp]),
    "kq_test_hold_copies": (ctypes.c_int, [ctypes.c_int]),
    "kq_status_str": (ctypes.c_char_p, [ctypes.c_int]),
}

_LIB = None


class KQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)}")


def lib() -> ctypes.CDLL:
    """The loaded libkq (loaded once)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libkq is not built ({LIB_PATH} missing); run __graft_entry__.build() "
                              "or python -m quantized_weight_matmul_q4_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def status_str(status: int) -> str:
    return lib().kq_status_str(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != KQ_OK:
        raise KQError(status, where)


def header_symbols() -> list[str]:
    """Names of the functions include/kq.h declares (for the ABI test)."""
    with open(os.path.join(INCLUDE, "kq.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"KQ_API\s+[\w\s\*]+?\b(kq_\w+)\s*\(", text)))
