"""CPU oracle for NVFP4 quantization and the block-scaled GEMM (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
legs of ``bench.py`` may import this package.  The CUDA path shares nothing with
it.  The arithmetic lives in ``nvfp4_oracle.c`` (plain C, single-threaded,
``-ffp-contract=off``; ``threads=`` runs the same per-row steps on several threads,
only to time the oracle on all host cores); this module only compiles it with gcc
and marshals numpy arrays through ctypes.  Each C function cites the passage of the news page
"NVIDIA NVFP4 paper: 4-bit pretrain hits FP8 parity (12B, 10T tokens)" it
follows, and marks every reading the page leaves open.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB = os.path.join(_HERE, "libnvfp4_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
RNE, SR = 0, 1
ROW, COL, TILE16 = 0, 1, 2
ERR_NONFINITE = 7

_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-fno-fast-math",
           "-Wall", "-Wno-unused-function"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no CUDA); rebuild when the source is newer."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".{os.getpid()}.tmp"
            subprocess.run(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    c = ctypes
    P = c.c_void_p
    sig = {
        "orc_e2m1_value": (c.c_double, [c.c_int]),
        "orc_e4m3_value": (c.c_double, [c.c_int]),
        "orc_e4m3_encode": (c.c_uint8, [c.c_float]),
        "orc_e2m1_encode_rne": (c.c_int, [c.c_float]),
        "orc_e2m1_encode_sr": (c.c_int, [c.c_float, c.c_uint32]),
        "orc_philox4x32_10": (None, [P, P, P]),
        "orc_sr_bits": (c.c_uint32, [c.c_uint64, c.c_uint32, c.c_uint32, c.c_uint64]),
        "orc_rht_sign_mask": (c.c_uint32, [c.c_uint64]),
        "orc_hadamard_stage_product": (None, [P]),
        "orc_rht16": (None, [P, c.c_uint32, P]),
        "orc_quantize": (c.c_int, [P, c.c_int, c.c_int64, c.c_int64, c.c_int64, c.c_int, c.c_int,
                                   c.c_int, c.c_uint64, c.c_uint32, c.c_uint64, P, P, P, P,
                                   c.c_int64, c.c_int64]),
        "orc_dequant": (None, [P, P, c.c_float, c.c_int64, c.c_int64, c.c_int, c.c_int64,
                               c.c_int64, P]),
        "orc_gemm_f64": (None, [P, P, c.c_int64, c.c_int64, c.c_int64, P]),
        "orc_quantize_mt": (c.c_int, [P, c.c_int, c.c_int64, c.c_int64, c.c_int64, c.c_int, c.c_int,
                                      c.c_int, c.c_uint64, c.c_uint32, c.c_uint64, P, P, P, P,
                                      c.c_int64, c.c_int64, c.c_int]),
        "orc_gemm_f64_mt": (None, [P, P, c.c_int64, c.c_int64, c.c_int64, P, c.c_int]),
        "orc_e4m3_encode_array": (None, [P, c.c_int64, P]),
        "orc_e2m1_encode_rne_array": (None, [P, c.c_int64, P]),
        "orc_e2m1_encode_sr_array": (None, [P, P, c.c_int64, P]),
        "orc_sr_bits_array": (None, [c.c_uint64, c.c_uint32, c.c_uint32, P, c.c_int64, P]),
        "orc_mx_scale_code": (c.c_uint8, [c.c_float]),
        "orc_mx_scale_value": (c.c_double, [c.c_int]),
        "orc_mx_quantize": (c.c_int, [P, c.c_int, c.c_int64, c.c_int64, c.c_int64, c.c_int, P, P]),
        "orc_mx_dequant": (None, [P, P, c.c_int64, c.c_int64, c.c_int64, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# --- codecs ------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return _load().orc_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return _load().orc_e4m3_value(int(code))


def e4m3_encode(v) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32).reshape(-1))
    out = np.empty(v.size, dtype=np.uint8)
    _load().orc_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e2m1_encode_rne(y) -> np.ndarray:
    y = np.ascontiguousarray(np.asarray(y, dtype=np.float32).reshape(-1))
    out = np.empty(y.size, dtype=np.uint8)
    _load().orc_e2m1_encode_rne_array(_ptr(y), y.size, _ptr(out))
    return out


def e2m1_encode_sr(y, r16) -> np.ndarray:
    y = np.ascontiguousarray(np.asarray(y, dtype=np.float32).reshape(-1))
    r = np.ascontiguousarray(np.broadcast_to(np.asarray(r16, dtype=np.uint32), y.shape))
    out = np.empty(y.size, dtype=np.uint8)
    _load().orc_e2m1_encode_sr_array(_ptr(y), _ptr(r), y.size, _ptr(out))
    return out


# --- random bits ---------------------------------------------------------------

def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    _load().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def sr_bits(seed: int, stream: int, offset: int, idx) -> np.ndarray:
    i = np.ascontiguousarray(np.asarray(idx, dtype=np.uint64).reshape(-1))
    out = np.empty(i.size, dtype=np.uint32)
    _load().orc_sr_bits_array(seed, stream, offset, _ptr(i), i.size, _ptr(out))
    return out


# --- RHT ---------------------------------------------------------------------------

def rht_sign_mask(seed: int) -> int:
    return int(_load().orc_rht_sign_mask(seed))


def hadamard_stage_product() -> np.ndarray:
    H = np.zeros(256, dtype=np.int32)
    _load().orc_hadamard_stage_product(_ptr(H))
    return H.reshape(16, 16)


def rht16(v, sign_mask: int) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32).reshape(16))
    y = np.empty(16, dtype=np.float32)
    _load().orc_rht16(_ptr(v), sign_mask, _ptr(y))
    return y


# --- quantize / dequant / GEMM --------------------------------------------------------

def quantize(x: np.ndarray, block: int, round_mode: int = RNE, rht: bool = False,
             sr_seed: int = 0, sr_offset: int = 0, rht_seed: int = 0,
             row_begin: int = 0, row_end: int = -1, ldx: int | None = None, threads: int = 1) -> dict:
    """Quantize ``x`` ([R, C] float32, or uint16 holding bf16 bits).

    Returns dict(codes, scales, s_dec, amax, rows, cols).  For ``block == COL``
    the operand is x^T: codes [C, R/2], scales [C, R/16].  For ``TILE16`` the
    scales are the [R/16, C/16] tile grid.  Rows outside [row_begin, row_end)
    of the operand are left zero.  ``threads`` > 1 splits the same per-row work among
    that many threads (identical results; for timing on all host cores).
    """
    if x.dtype == np.float32:
        dtype = F32
    elif x.dtype == np.uint16:
        dtype = BF16
    else:
        raise TypeError("oracle.quantize takes float32 or uint16 (bf16 bits)")
    x = np.ascontiguousarray(x) if ldx is None else x
    R, C = x.shape
    ld = C if ldx is None else ldx
    rows, cols = (C, R) if block == COL else (R, C)
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    if block == TILE16:
        scales = np.zeros((rows // 16, cols // 16), dtype=np.uint8)
    else:
        scales = np.zeros((rows, cols // 16), dtype=np.uint8)
    s_dec = np.zeros(1, dtype=np.float32)
    amax = np.zeros(1, dtype=np.float32)
    args = (_ptr(x), dtype, R, C, ld, block, round_mode, int(bool(rht)), sr_seed, sr_offset, rht_seed,
            _ptr(codes), _ptr(scales), _ptr(s_dec), _ptr(amax), row_begin, row_end)
    st = _load().orc_quantize(*args) if threads <= 1 else _load().orc_quantize_mt(*args, int(threads))
    if st == ERR_NONFINITE:
        raise FloatingPointError("non-finite tensor amax")
    if st != 0:
        raise ValueError(f"oracle quantize rejected the arguments (status {st})")
    return dict(codes=codes, scales=scales, s_dec=float(s_dec[0]), amax=float(amax[0]),
                rows=rows, cols=cols, block=block)


def dequant(q: dict, row_begin: int = 0, row_end: int | None = None) -> np.ndarray:
    rows, cols = q["rows"], q["cols"]
    row_end = rows if row_end is None else row_end
    out = np.empty((row_end - row_begin, cols), dtype=np.float64)
    codes = np.ascontiguousarray(q["codes"])
    scales = np.ascontiguousarray(q["scales"])
    _load().orc_dequant(_ptr(codes), _ptr(scales), q["s_dec"], rows, cols,
                        int(q["block"] == TILE16), row_begin, row_end, _ptr(out))
    return out


def gemm_f64(A: np.ndarray, B: np.ndarray, threads: int = 1) -> np.ndarray:
    """C = A . B^T in fp64 (plain dot products); ``threads`` > 1 splits C's rows."""
    A = np.ascontiguousarray(A, dtype=np.float64)
    B = np.ascontiguousarray(B, dtype=np.float64)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2
    C = np.empty((M, N), dtype=np.float64)
    if threads <= 1:
        _load().orc_gemm_f64(_ptr(A), _ptr(B), M, N, K, _ptr(C))
    else:
        _load().orc_gemm_f64_mt(_ptr(A), _ptr(B), M, N, K, _ptr(C), int(threads))
    return C


def host_cores() -> int:
    """Cores this process may run on (sched_getaffinity), for the threaded timings."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


# --- squared ReLU of the dense MLP block (plain numpy float32) -------------------------

def _bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bits (finite inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def sqrelu_forward(h_bits: np.ndarray) -> np.ndarray:
    """a = relu(h)^2 with relu(h) = h if h > 0 else +0; bf16 bits in and out."""
    h = _bf16_to_f32(h_bits)
    r = np.where(h > 0, h, np.float32(0)).astype(np.float32)
    return _f32_to_bf16((r * r).astype(np.float32))


def sqrelu_backward(h_bits: np.ndarray, da_bits: np.ndarray) -> np.ndarray:
    """dh = da * (2 relu(h)); bf16 bits in and out."""
    h = _bf16_to_f32(h_bits)
    da = _bf16_to_f32(da_bits)
    t = np.where(h > 0, (np.float32(2) * h).astype(np.float32), np.float32(0)).astype(np.float32)
    return _f32_to_bf16((da * t).astype(np.float32))


# --- MXFP4 (the comparison format: 1x32 blocks, power-of-two scales, no tensor scale) ---

def mx_scale_code(amax: float) -> int:
    return int(_load().orc_mx_scale_code(float(amax)))


def mx_scale_value(code: int) -> float:
    return float(_load().orc_mx_scale_value(int(code)))


def mx_quantize(x: np.ndarray, col: bool = False) -> dict:
    """MXFP4 of ``x`` ([R, C] float32 or uint16 bf16 bits): operand x (or x^T with
    ``col``), 1x32 blocks along the operand's rows.  dict(codes, scales, rows, cols)."""
    if x.dtype == np.float32:
        dtype = F32
    elif x.dtype == np.uint16:
        dtype = BF16
    else:
        raise TypeError("oracle.mx_quantize takes float32 or uint16 (bf16 bits)")
    x = np.ascontiguousarray(x)
    R, C = x.shape
    rows, cols = (C, R) if col else (R, C)
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    scales = np.zeros((rows, cols // 32), dtype=np.uint8)
    st = _load().orc_mx_quantize(_ptr(x), dtype, R, C, C, int(bool(col)), _ptr(codes), _ptr(scales))
    if st == ERR_NONFINITE:
        raise FloatingPointError("non-finite input")
    if st != 0:
        raise ValueError(f"oracle mx_quantize rejected the arguments (status {st})")
    return dict(codes=codes, scales=scales, rows=rows, cols=cols)


def mx_dequant(q: dict, row_begin: int = 0, row_end: int | None = None) -> np.ndarray:
    rows, cols = q["rows"], q["cols"]
    row_end = rows if row_end is None else row_end
    out = np.empty((row_end - row_begin, cols), dtype=np.float64)
    _load().orc_mx_dequant(_ptr(np.ascontiguousarray(q["codes"])), _ptr(np.ascontiguousarray(q["scales"])),
                           cols, row_begin, row_end, _ptr(out))
    return out
