"""Torch-facing wrappers of the C ABI (include/nvfp4.h): argument marshalling only.

Every function takes CUDA tensors, allocates outputs with torch, and launches
the library's kernels on ``torch.cuda.current_stream()``.  Host-side argument
errors raise :class:`NVFP4Error` before anything is launched; device-side errors
(a non-finite tensor, a timed-out pipeline wait) land in the per-device status
word read by :func:`status_query`.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib as L
from ._lib import NVFP4Error

_DT = {torch.float32: L.F32, torch.bfloat16: L.BF16}


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _check_2d(x: torch.Tensor, name: str) -> None:
    if not x.is_cuda:
        raise NVFP4Error(L.ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
    if x.dim() != 2 or (x.shape[1] > 1 and x.stride(1) != 1):
        raise NVFP4Error(L.ERR_INVALID_ARG, f"{name} must be 2-D with unit column stride")
    if x.dtype not in _DT:
        raise NVFP4Error(L.ERR_INVALID_ARG, f"{name} must be float32 or bfloat16")


# ----------------------------------------------------------------------------- status

_status: dict = {}


def dev_status(device=None) -> torch.Tensor:
    """The device status word (uint32 stored in an int32 tensor) for ``device``."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else torch.device(device).index)
    t = _status.get(dev.index)
    if t is None:
        t = torch.zeros(4, dtype=torch.int32, device=dev)
        _status[dev.index] = t
    return t


def reset_status(device=None) -> None:
    dev_status(device).zero_()


def status_query(device=None) -> int:
    """Synchronises the current stream and returns the device status (0 = ok)."""
    return int(L.lib().nvfp4_status_query(dev_status(device).data_ptr(), _stream()))


# ----------------------------------------------------------------------------- workspace

_ws: dict = {}


def _workspace(nbytes: int) -> torch.Tensor:
    key = (torch.cuda.current_device(), _stream())
    t = _ws.get(key)
    if t is None or t.numel() < nbytes:
        t = torch.empty(max(nbytes, 1 << 16), dtype=torch.uint8, device="cuda")
        _ws[key] = t
    return t


def scales_mma_bytes(rows: int, cols: int) -> int:
    return int(L.lib().nvfp4_scales_mma_bytes(rows, cols))


# ----------------------------------------------------------------------------- quantized operand

@dataclass
class QTensor:
    """A quantized operand of logical shape [rows, cols] (16-element blocks along cols)."""
    codes: torch.Tensor                       # uint8 [rows, cols/2]
    scales: Optional[torch.Tensor]            # uint8 [rows, cols/16] (TILE16: [rows/16, cols/16])
    scales_mma: Optional[torch.Tensor]        # uint8, tensor-core tile layout
    s_dec: torch.Tensor                       # float32 [4]; element 0 is the tensor decode scale
    rows: int
    cols: int
    block: int
    codes_t: Optional[torch.Tensor] = None    # TILE16 only: codes of the transpose
    scales_mma_t: Optional[torch.Tensor] = None

    def c_struct(self) -> L.QTensorC:
        return L.QTensorC(_ptr(self.codes), _ptr(self.scales), _ptr(self.scales_mma), _ptr(self.s_dec),
                          _ptr(self.codes_t), _ptr(self.scales_mma_t), self.rows, self.cols)

    def transposed(self) -> "QTensor":
        """W^T as an operand (TILE16 quantization with the transposed copy)."""
        if self.codes_t is None or self.scales_mma_t is None:
            raise NVFP4Error(L.ERR_INVALID_ARG, "no transposed copy was written")
        return QTensor(self.codes_t, None, self.scales_mma_t, self.s_dec, self.cols, self.rows, self.block)


def _alloc_q(R: int, C: int, block: int, dev, scales: bool, scales_mma: bool, transpose: bool) -> QTensor:
    rows, cols = (C, R) if block == L.COL else (R, C)
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
    sc = None
    if scales:
        shape = (rows // 16, cols // 16) if block == L.TILE16 else (rows, cols // 16)
        sc = torch.empty(shape, dtype=torch.uint8, device=dev)
    smma = torch.empty(max(scales_mma_bytes(rows, cols), 16), dtype=torch.uint8, device=dev) if scales_mma else None
    s_dec = torch.empty(4, dtype=torch.float32, device=dev)
    codes_t = smma_t = None
    if block == L.TILE16 and transpose:
        codes_t = torch.empty((cols, rows // 2), dtype=torch.uint8, device=dev)
        smma_t = torch.empty(max(scales_mma_bytes(cols, rows), 16), dtype=torch.uint8, device=dev)
    return QTensor(codes, sc, smma, s_dec, rows, cols, block, codes_t, smma_t)


def _params(block, round, rht, sr_seed, sr_offset, rht_seed) -> L.QParams:
    return L.QParams(block, round, int(bool(rht)), sr_offset & 0xFFFFFFFF, sr_seed & (2**64 - 1),
                     rht_seed & (2**64 - 1))


def quantize(x: torch.Tensor, block: int = L.ROW, round: int = L.RNE, rht: bool = False,
             sr_seed: int = 0, sr_offset: int = 0, rht_seed: int = 0, scales: bool = True,
             scales_mma: bool = True, transpose: bool = True) -> QTensor:
    """Quantize x [R, C] (float32 / bfloat16, CUDA) to NVFP4 with the library's kernels."""
    _check_2d(x, "x")
    R, C = x.shape
    q = _alloc_q(R, C, block, x.device, scales, scales_mma, transpose)
    params = _params(block, round, rht, sr_seed, sr_offset, rht_seed)
    qc = q.c_struct()
    lib = L.lib()
    ws_bytes = int(lib.nvfp4_quantize_workspace_bytes(R, C, ctypes.byref(params)))
    ws = _workspace(ws_bytes)
    ld = x.stride(0) if R > 1 else max(C, 1)
    st = lib.nvfp4_quantize(_ptr(x), _DT[x.dtype], R, C, ld, ctypes.byref(params), ctypes.byref(qc),
                            ws.data_ptr(), ws.numel(), dev_status(x.device).data_ptr(), _stream())
    L.check(st, "nvfp4_quantize")
    return q


def quantize_dual(x: torch.Tensor, row_round: int = L.RNE, col_round: int = L.RNE, rht: bool = True,
                  sr_seed: int = 0, sr_offset: int = 0, rht_seed: int = 0, scales: bool = True,
                  scales_mma: bool = True, col_sr_seed: Optional[int] = None, col_sr_offset: Optional[int] = None,
                  pre: Optional[str] = None, maxima: Optional[torch.Tensor] = None):
    """Both training quantizations of x [R, C] from one amax read: the 1x16 row
    operand [R, C] and the 1x16 column operand [C, R] (RHT along R when ``rht``).
    Identical to two ``quantize`` calls with the same parameters; the column
    operand's SR seed / offset default to the row's.  ``pre="sqrelu"`` quantizes
    relu(x)^2 (bf16 x) without storing it, identical to ``sqrelu_forward`` first.
    ``maxima``: the partial maxima a producing GEMM left for this x with the same
    ``rht_seed`` (``gemm_sqrelu_maxima`` with ``pre="sqrelu"``, ``gemm_sqrelu_backward(...,
    maxima=True)`` without); the amax read is then skipped."""
    _check_2d(x, "x")
    R, C = x.shape
    qr = _alloc_q(R, C, L.ROW, x.device, scales, scales_mma, False)
    qc = _alloc_q(R, C, L.COL, x.device, scales, scales_mma, False)
    pr = _params(L.ROW, row_round, False, sr_seed, sr_offset, rht_seed)
    pc = _params(L.COL, col_round, rht, sr_seed if col_sr_seed is None else col_sr_seed,
                 sr_offset if col_sr_offset is None else col_sr_offset, rht_seed)
    a, b = qr.c_struct(), qc.c_struct()
    lib = L.lib()
    ws = _workspace(int(lib.nvfp4_quantize_dual_workspace_bytes(R, C)))
    ld = x.stride(0) if R > 1 else max(C, 1)
    if pre not in (None, "sqrelu"):
        raise ValueError(f"unknown pre transform {pre!r}")
    if maxima is not None:
        fn = lib.nvfp4_quantize_dual_sqrelu_premax if pre == "sqrelu" else lib.nvfp4_quantize_dual_premax
        st = fn(_ptr(x), _DT[x.dtype], R, C, ld, ctypes.byref(pr), ctypes.byref(a), ctypes.byref(pc), ctypes.byref(b),
                _ptr(maxima), maxima.numel() * maxima.element_size(), dev_status(x.device).data_ptr(), _stream())
        L.check(st, "nvfp4_quantize_dual_sqrelu_premax" if pre else "nvfp4_quantize_dual_premax")
        return qr, qc
    fn = lib.nvfp4_quantize_dual_sqrelu if pre == "sqrelu" else lib.nvfp4_quantize_dual
    st = fn(_ptr(x), _DT[x.dtype], R, C, ld, ctypes.byref(pr), ctypes.byref(a), ctypes.byref(pc), ctypes.byref(b),
            ws.data_ptr(), ws.numel(), dev_status(x.device).data_ptr(), _stream())
    L.check(st, "nvfp4_quantize_dual_sqrelu" if pre else "nvfp4_quantize_dual")
    return qr, qc


def quantize_weight(W: torch.Tensor) -> QTensor:
    """Weights: 16x16 2D blocks, RNE, with the transposed copy for Dgrad [page ¶2]."""
    return quantize(W, L.TILE16, L.RNE, transpose=True)


_gemm_ws = {}


def _gemm_workspace(device) -> torch.Tensor:
    """The split-tail workspace of ``gemm(..., split_tail=True)`` for this device and stream:
    zero-filled once; every call leaves it zeroed (after a device error, call
    ``reset_gemm_workspaces``)."""
    dev = torch.device(device)
    key = (dev.index, _stream())
    t = _gemm_ws.get(key)
    if t is None:
        nbytes = int(L.lib().nvfp4_gemm_workspace_bytes(dev.index))
        if nbytes == 0:
            raise NVFP4Error(L.ERR_CUDA, "cannot size the GEMM workspace for this device")
        t = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        _gemm_ws[key] = t
    return t


def reset_gemm_workspaces() -> None:
    """Zero-fill every cached split-tail workspace (needed after a GEMM reported a device error)."""
    for t in _gemm_ws.values():
        t.zero_()


def gemm(A: QTensor, B: QTensor, out_dtype=torch.bfloat16, out: Optional[torch.Tensor] = None,
         split_tail: bool = False) -> torch.Tensor:
    """D[M, N] = dequant(A) . dequant(B)^T on the tcgen05 block-scaled FP4 tensor cores.
    With ``split_tail`` (nvfp4_gemm_ws), the tiles of the last partial wave are cut in two along
    K over more SM pairs (deterministic; those tiles' fp32 sums are grouped differently)."""
    M, N = A.rows, B.rows
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=A.codes.device)
    _check_2d(out, "out")
    a, b = A.c_struct(), B.c_struct()
    if split_tail:
        ws = _gemm_workspace(out.device)
        st = L.lib().nvfp4_gemm_ws(ctypes.byref(a), ctypes.byref(b), _ptr(out), _DT[out.dtype], out.stride(0),
                                   _ptr(ws), ws.numel(), dev_status(out.device).data_ptr(), _stream())
        L.check(st, "nvfp4_gemm_ws")
        return out
    st = L.lib().nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), _ptr(out), _DT[out.dtype], out.stride(0),
                            dev_status(out.device).data_ptr(), _stream())
    L.check(st, "nvfp4_gemm")
    return out


# ----------------------------------------------------------------------------- MXFP4 comparison format

@dataclass
class MXTensor:
    """An MXFP4 operand of logical shape [rows, cols]: 32-element blocks along cols,
    UE8M0 power-of-two scales, no tensor scale."""
    codes: torch.Tensor                       # uint8 [rows, cols/2]
    scales: Optional[torch.Tensor]            # uint8 [rows, cols/32]
    scales_mma: Optional[torch.Tensor]        # uint8, 1 KB-tile layout
    rows: int
    cols: int

    def c_struct(self) -> L.QTensorC:
        return L.QTensorC(_ptr(self.codes), _ptr(self.scales), _ptr(self.scales_mma), None, None, None,
                          self.rows, self.cols)


def mx_scales_mma_bytes(rows: int, cols: int) -> int:
    return int(L.lib().nvfp4_mx_scales_mma_bytes(rows, cols))


def mx_quantize(x: torch.Tensor, col: bool = False, scales: bool = True, scales_mma: bool = True) -> MXTensor:
    """MXFP4 quantization of x [R, C] (blocks along C), or of x^T [C, R] with ``col``."""
    _check_2d(x, "x")
    R, C = x.shape
    rows, cols = (C, R) if col else (R, C)
    dev = x.device
    q = MXTensor(torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev),
                 torch.empty((rows, cols // 32), dtype=torch.uint8, device=dev) if scales else None,
                 torch.empty(max(mx_scales_mma_bytes(rows, cols), 16), dtype=torch.uint8, device=dev)
                 if scales_mma else None, rows, cols)
    qc = q.c_struct()
    ld = x.stride(0) if R > 1 else max(C, 1)
    st = L.lib().nvfp4_mx_quantize(_ptr(x), _DT[x.dtype], R, C, ld, int(bool(col)), ctypes.byref(qc), _stream())
    L.check(st, "nvfp4_mx_quantize")
    return q


def mx_gemm(A: MXTensor, B: MXTensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """D[M, N] = dequant(A) . dequant(B)^T for MXFP4 operands (bf16 out) on the FP4 tensor cores."""
    M, N = A.rows, B.rows
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.codes.device)
    _check_2d(out, "out")
    a, b = A.c_struct(), B.c_struct()
    st = L.lib().nvfp4_mx_gemm(ctypes.byref(a), ctypes.byref(b), _ptr(out), _DT[out.dtype], out.stride(0),
                               dev_status(out.device).data_ptr(), _stream())
    L.check(st, "nvfp4_mx_gemm")
    return out


def _maxima_buffer(device) -> torch.Tensor:
    """A partial-maxima buffer for the *_maxima GEMMs on ``device`` (sized by its SM count)."""
    nbytes = int(L.lib().nvfp4_sqrelu_maxima_bytes(torch.device(device).index))
    if nbytes == 0:
        raise NVFP4Error(L.ERR_CUDA, "cannot size the maxima buffer for this device")
    return torch.empty(nbytes // 4, dtype=torch.int32, device=device)


def gemm_sqrelu_maxima(A: QTensor, B: QTensor, rht_seed: int = 0, out: Optional[torch.Tensor] = None):
    """H = dequant(A) . dequant(B)^T in bf16 (as ``gemm`` stores it), plus the partial tensor
    maxima of relu(H)^2 that ``quantize_dual(H, ..., pre="sqrelu", maxima=m)`` needs, computed
    in the GEMM's epilogue (RHT signs from ``rht_seed``).  Returns (H, m)."""
    M, N = A.rows, B.rows
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.codes.device)
    _check_2d(out, "out")
    lib = L.lib()
    m = _maxima_buffer(out.device)
    a, b = A.c_struct(), B.c_struct()
    st = lib.nvfp4_gemm_sqrelu_maxima(ctypes.byref(a), ctypes.byref(b), _ptr(out), out.stride(0) if M > 1 else N,
                                      rht_seed & (2**64 - 1), _ptr(m), m.numel() * 4, dev_status(out.device).data_ptr(),
                                      _stream())
    L.check(st, "nvfp4_gemm_sqrelu_maxima")
    return out, m


def gemm_sqrelu_backward(A: QTensor, B: QTensor, H: torch.Tensor, out: Optional[torch.Tensor] = None,
                         maxima: bool = False, rht_seed: int = 0):
    """dH = dA * 2 relu(H) with dA = dequant(A) . dequant(B)^T in bf16 -- the Dgrad GEMM of a
    squared-ReLU MLP with the activation's backward in its epilogue (dA is never stored);
    bit for bit ``sqrelu_backward(H, gemm(A, B, torch.bfloat16))``.  H: bf16 [M, N].  With
    ``maxima`` the epilogue also leaves dH's tensor maxima for ``quantize_dual(dH, ...,
    maxima=m)`` (RHT signs from ``rht_seed``) and (dH, m) is returned."""
    M, N = A.rows, B.rows
    _check_2d(H, "H")
    if H.dtype != torch.bfloat16 or tuple(H.shape) != (M, N):
        raise NVFP4Error(L.ERR_INVALID_ARG, f"H must be bfloat16 [{M}, {N}]")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.codes.device)
    _check_2d(out, "out")
    a, b = A.c_struct(), B.c_struct()
    lib = L.lib()
    ldh, ldd = H.stride(0) if M > 1 else N, out.stride(0) if M > 1 else N
    if maxima:
        m = _maxima_buffer(out.device)
        st = lib.nvfp4_gemm_sqrelu_bwd_maxima(ctypes.byref(a), ctypes.byref(b), _ptr(H), ldh, _ptr(out), ldd,
                                              rht_seed & (2**64 - 1), _ptr(m), m.numel() * 4,
                                              dev_status(out.device).data_ptr(), _stream())
        L.check(st, "nvfp4_gemm_sqrelu_bwd_maxima")
        return out, m
    st = lib.nvfp4_gemm_sqrelu_bwd(ctypes.byref(a), ctypes.byref(b), _ptr(H), ldh, _ptr(out), ldd,
                                   dev_status(out.device).data_ptr(), _stream())
    L.check(st, "nvfp4_gemm_sqrelu_bwd")
    return out


def _linear_ws(M: int, N: int, K: int) -> torch.Tensor:
    return _workspace(int(L.lib().nvfp4_linear_workspace_bytes(M, N, K)))


def linear_fprop(X: torch.Tensor, Wq: QTensor, out_dtype=torch.bfloat16) -> torch.Tensor:
    """Y[M, N] = X . W^T; X quantized 1x16 RNE inside the call."""
    _check_2d(X, "X")
    M, K = X.shape
    N = Wq.rows
    Y = torch.empty((M, N), dtype=out_dtype, device=X.device)
    ws = _linear_ws(M, N, K)
    w = Wq.c_struct()
    st = L.lib().nvfp4_linear_fprop(_ptr(X), _DT[X.dtype], M, K, X.stride(0), ctypes.byref(w), _ptr(Y),
                                    _DT[out_dtype], Y.stride(0), ws.data_ptr(), ws.numel(),
                                    dev_status(X.device).data_ptr(), _stream())
    L.check(st, "nvfp4_linear_fprop")
    return Y


def linear_dgrad(dY: torch.Tensor, Wq: QTensor, sr_seed: int = 0, sr_offset: int = 0,
                 out_dtype=torch.bfloat16) -> torch.Tensor:
    """dX[M, K] = dY . W; dY quantized 1x16 with stochastic rounding inside the call."""
    _check_2d(dY, "dY")
    M, N = dY.shape
    K = Wq.cols
    dX = torch.empty((M, K), dtype=out_dtype, device=dY.device)
    ws = _linear_ws(M, N, K)
    w = Wq.c_struct()
    st = L.lib().nvfp4_linear_dgrad(_ptr(dY), _DT[dY.dtype], M, N, dY.stride(0), ctypes.byref(w),
                                    sr_seed & (2**64 - 1), sr_offset & 0xFFFFFFFF, _ptr(dX), _DT[out_dtype],
                                    dX.stride(0), ws.data_ptr(), ws.numel(), dev_status(dY.device).data_ptr(),
                                    _stream())
    L.check(st, "nvfp4_linear_dgrad")
    return dX


def linear_wgrad(dY: torch.Tensor, X: torch.Tensor, sr_seed: int = 0, sr_offset: int = 0, rht_seed: int = 0,
                 out_dtype=torch.bfloat16) -> torch.Tensor:
    """dW[N, K] = dY^T . X; both quantized 1x16 along M after the shared-sign RHT."""
    _check_2d(dY, "dY")
    _check_2d(X, "X")
    M, N = dY.shape
    K = X.shape[1]
    if X.shape[0] != M:
        raise NVFP4Error(L.ERR_SHAPE, "dY and X disagree on M")
    dW = torch.empty((N, K), dtype=out_dtype, device=dY.device)
    ws = _linear_ws(M, N, K)
    st = L.lib().nvfp4_linear_wgrad(_ptr(dY), _DT[dY.dtype], dY.stride(0), _ptr(X), _DT[X.dtype], X.stride(0),
                                    M, N, K, sr_seed & (2**64 - 1), sr_offset & 0xFFFFFFFF, rht_seed & (2**64 - 1),
                                    _ptr(dW), _DT[out_dtype], dW.stride(0), ws.data_ptr(), ws.numel(),
                                    dev_status(dY.device).data_ptr(), _stream())
    L.check(st, "nvfp4_linear_wgrad")
    return dW


def sqrelu_forward(h: torch.Tensor) -> torch.Tensor:
    """a = relu(h)^2 (bf16, contiguous)."""
    if h.dtype != torch.bfloat16 or not h.is_contiguous() or not h.is_cuda:
        raise NVFP4Error(L.ERR_INVALID_ARG, "h must be a contiguous CUDA bf16 tensor")
    a = torch.empty_like(h)
    L.check(L.lib().nvfp4_sqrelu_forward(h.data_ptr(), a.data_ptr(), h.numel(), _stream()), "nvfp4_sqrelu_forward")
    return a


def sqrelu_backward(h: torch.Tensor, da: torch.Tensor) -> torch.Tensor:
    """dh = da * 2 relu(h) (bf16, contiguous)."""
    for t, n in ((h, "h"), (da, "da")):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
            raise NVFP4Error(L.ERR_INVALID_ARG, f"{n} must be a contiguous CUDA bf16 tensor")
    if h.shape != da.shape:
        raise NVFP4Error(L.ERR_SHAPE, "h and da differ in shape")
    dh = torch.empty_like(h)
    L.check(L.lib().nvfp4_sqrelu_backward(h.data_ptr(), da.data_ptr(), dh.data_ptr(), h.numel(), _stream()),
            "nvfp4_sqrelu_backward")
    return dh
