"""ctypes view of the C ABI in include/nvfp4.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libnvfp4_gb300.so")

OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_ALIGNMENT, ERR_WORKSPACE, ERR_UNSUPPORTED, ERR_CUDA, ERR_NONFINITE, ERR_TIMEOUT = range(9)
F32, BF16 = 0, 1
RNE, SR = 0, 1
ROW, COL, TILE16 = 0, 1, 2

# every symbol include/nvfp4.h declares
EXPORTS = [
    "nvfp4_scales_mma_bytes", "nvfp4_quantize_workspace_bytes", "nvfp4_quantize", "nvfp4_quantize_noalloc",
    "nvfp4_quantize_dual_workspace_bytes", "nvfp4_quantize_dual", "nvfp4_quantize_dual_sqrelu",
    "nvfp4_gemm", "nvfp4_gemm_workspace_bytes", "nvfp4_gemm_ws",
    "nvfp4_linear_workspace_bytes", "nvfp4_linear_fprop", "nvfp4_linear_dgrad", "nvfp4_linear_wgrad",
    "nvfp4_status_query", "nvfp4_status_string", "nvfp4_set_wait_timeout_ns", "nvfp4_debug_e4m3",
    "nvfp4_debug_e2m1", "nvfp4_debug_philox", "nvfp4_selftest_wait_timeout", "nvfp4_gemm_force_path",
    "nvfp4_sqrelu_forward", "nvfp4_sqrelu_backward",
    "nvfp4_mx_scales_mma_bytes", "nvfp4_mx_quantize", "nvfp4_mx_gemm", "nvfp4_gemm_sqrelu_bwd",
    "nvfp4_sqrelu_maxima_bytes", "nvfp4_gemm_sqrelu_maxima", "nvfp4_quantize_dual_sqrelu_premax",
    "nvfp4_gemm_sqrelu_bwd_maxima", "nvfp4_quantize_dual_premax",
]


class QParams(ctypes.Structure):
    _fields_ = [("block", ctypes.c_int32), ("round", ctypes.c_int32), ("rht", ctypes.c_int32),
                ("sr_offset", ctypes.c_uint32), ("sr_seed", ctypes.c_uint64), ("rht_seed", ctypes.c_uint64)]


class QTensorC(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("scales_mma", ctypes.c_void_p),
                ("s_dec", ctypes.c_void_p), ("codes_t", ctypes.c_void_p), ("scales_mma_t", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})" if what else status_string(status))


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded library.  Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        c = ctypes
        P, I64, I32, U32, U64, SZ = c.c_void_p, c.c_int64, c.c_int32, c.c_uint32, c.c_uint64, c.c_size_t
        QP, QT = c.POINTER(QParams), c.POINTER(QTensorC)
        sigs = {
            "nvfp4_scales_mma_bytes": (SZ, [I64, I64]),
            "nvfp4_quantize_workspace_bytes": (SZ, [I64, I64, QP]),
            "nvfp4_quantize": (I32, [P, I32, I64, I64, I64, QP, QT, P, SZ, P, P]),
            "nvfp4_quantize_noalloc": (I32, [P, I32, I64, I64, I64, QP, QT, P, P]),
            "nvfp4_quantize_dual_workspace_bytes": (SZ, [I64, I64]),
            "nvfp4_quantize_dual": (I32, [P, I32, I64, I64, I64, QP, QT, QP, QT, P, SZ, P, P]),
            "nvfp4_quantize_dual_sqrelu": (I32, [P, I32, I64, I64, I64, QP, QT, QP, QT, P, SZ, P, P]),
            "nvfp4_gemm": (I32, [QT, QT, P, I32, I64, P, P]),
            "nvfp4_gemm_workspace_bytes": (SZ, [I32]),
            "nvfp4_gemm_ws": (I32, [QT, QT, P, I32, I64, P, SZ, P, P]),
            "nvfp4_linear_workspace_bytes": (SZ, [I64, I64, I64]),
            "nvfp4_linear_fprop": (I32, [P, I32, I64, I64, I64, QT, P, I32, I64, P, SZ, P, P]),
            "nvfp4_linear_dgrad": (I32, [P, I32, I64, I64, I64, QT, U64, U32, P, I32, I64, P, SZ, P, P]),
            "nvfp4_linear_wgrad": (I32, [P, I32, I64, P, I32, I64, I64, I64, I64, U64, U32, U64, P, I32, I64,
                                         P, SZ, P, P]),
            "nvfp4_status_query": (I32, [P, P]),
            "nvfp4_status_string": (c.c_char_p, [I32]),
            "nvfp4_set_wait_timeout_ns": (None, [U64]),
            "nvfp4_debug_e4m3": (I32, [P, I64, P, P]),
            "nvfp4_debug_e2m1": (I32, [P, P, I64, I32, I32, P, P]),
            "nvfp4_debug_philox": (I32, [P, I64, U64, P, P]),
            "nvfp4_selftest_wait_timeout": (I32, [U64, P, P]),
            "nvfp4_gemm_force_path": (None, [I32]),
            "nvfp4_sqrelu_forward": (I32, [P, P, I64, P]),
            "nvfp4_sqrelu_backward": (I32, [P, P, P, I64, P]),
            "nvfp4_mx_scales_mma_bytes": (SZ, [I64, I64]),
            "nvfp4_mx_quantize": (I32, [P, I32, I64, I64, I64, I32, QT, P]),
            "nvfp4_mx_gemm": (I32, [QT, QT, P, I32, I64, P, P]),
            "nvfp4_gemm_sqrelu_bwd": (I32, [QT, QT, P, I64, P, I64, P, P]),
            "nvfp4_sqrelu_maxima_bytes": (SZ, [I32]),
            "nvfp4_gemm_sqrelu_maxima": (I32, [QT, QT, P, I64, U64, P, SZ, P, P]),
            "nvfp4_quantize_dual_sqrelu_premax": (I32, [P, I32, I64, I64, I64, QP, QT, QP, QT, P, SZ, P, P]),
            "nvfp4_gemm_sqrelu_bwd_maxima": (I32, [QT, QT, P, I64, P, I64, U64, P, SZ, P, P]),
            "nvfp4_quantize_dual_premax": (I32, [P, I32, I64, I64, I64, QP, QT, QP, QT, P, SZ, P, P]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().nvfp4_status_string(int(status)).decode()


def check(status: int, what: str = "") -> None:
    if status != OK:
        raise NVFP4Error(status, what)
