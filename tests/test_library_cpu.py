"""Host-side checks of the C-ABI library that need no GPU: it loads, it exports
every symbol include/nvfp4.h declares, and argument errors come back as status
codes before anything touches CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build_library()
    from nvfp4_bit_quantized_gb300 import _lib
    return _lib


def test_exports_match_header(lib):
    hdr = open(os.path.join(ROOT, "include", "nvfp4.h")).read()
    declared = set(re.findall(r"NVFP4_API\s+[\w\s\*]+?\b(nvfp4_\w+)\s*\(", hdr))
    assert declared == set(lib.EXPORTS)
    L = lib.lib()
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings(lib):
    assert lib.status_string(0) == "ok"
    for s in range(1, 9):
        assert lib.status_string(s) not in ("ok", "unknown status")
    assert lib.status_string(99) == "unknown status"


def test_scale_layout_sizes(lib):
    L = lib.lib()
    assert L.nvfp4_scales_mma_bytes(128, 256) == 2048
    assert L.nvfp4_scales_mma_bytes(129, 256) == 4096
    assert L.nvfp4_scales_mma_bytes(8192, 5120) == 64 * 20 * 2048
    assert L.nvfp4_scales_mma_bytes(0, 256) == 0
    assert L.nvfp4_linear_workspace_bytes(8192, 20480, 5120) > 8192 * 20480 // 2


def _qp(lib, block=0, rnd=0, rht=0):
    return lib.QParams(block, rnd, rht, 0, 0, 0)


def test_quantize_rejects_bad_arguments_without_launching(lib):
    L = lib.lib()
    fake = ctypes.c_void_p(0x1000)          # never dereferenced: validation fails first
    sdec = ctypes.c_void_p(0x2000)
    q = lib.QTensorC(0x1000, 0x1000, None, sdec.value, None, None, 32, 64)
    ws = 4096 * 4
    cases = [
        (dict(dtype=5), lib.ERR_INVALID_ARG),                       # bad dtype
        (dict(block=7), lib.ERR_INVALID_ARG),                       # bad block
        (dict(rht=1), lib.ERR_INVALID_ARG),                         # RHT needs column blocks
        (dict(C=40, cols=40), lib.ERR_SHAPE),                       # C % 16
        (dict(rows=31), lib.ERR_SHAPE),                             # output shape mismatch
        (dict(ld=50), lib.ERR_SHAPE),                               # ldx < C
        (dict(x=0x1008), lib.ERR_ALIGNMENT),                        # misaligned input
        (dict(ws=16), lib.ERR_WORKSPACE),                           # too small workspace
    ]
    for kw, expect in cases:
        p = _qp(lib, kw.get("block", 0), 0, kw.get("rht", 0))
        qq = lib.QTensorC(q.codes, q.scales, None, q.s_dec, None, None, kw.get("rows", 32), kw.get("cols", 64))
        st = L.nvfp4_quantize(kw.get("x", fake.value), kw.get("dtype", lib.BF16), 32, kw.get("C", 64),
                              kw.get("ld", 64), ctypes.byref(p), ctypes.byref(qq), 0x3000, kw.get("ws", ws),
                              None, None)
        assert st == expect, (kw, st)
    st = L.nvfp4_quantize(fake, lib.BF16, 32, 64, 64, None, ctypes.byref(q), 0x3000, ws, None, None)
    assert st == lib.ERR_INVALID_ARG
    # the squared-ReLU dual quantization takes bf16 only
    pr, pc = _qp(lib, 0, 0, 0), _qp(lib, 1, 0, 1)
    qr = lib.QTensorC(0x1000, 0x1000, None, sdec.value, None, None, 32, 64)
    qc = lib.QTensorC(0x1000, 0x1000, None, sdec.value, None, None, 64, 32)
    st = L.nvfp4_quantize_dual_sqrelu(fake, lib.F32, 32, 64, 64, ctypes.byref(pr), ctypes.byref(qr), ctypes.byref(pc),
                                      ctypes.byref(qc), 0x3000, 2 * ws, None, None)
    assert st == lib.ERR_UNSUPPORTED


def test_gemm_and_linear_reject_bad_arguments(lib):
    L = lib.lib()
    A = lib.QTensorC(0x1000, None, 0x1000, 0x2000, None, None, 128, 256)
    B = lib.QTensorC(0x1000, None, 0x1000, 0x2000, None, None, 256, 128)     # K mismatch
    assert L.nvfp4_gemm(ctypes.byref(A), ctypes.byref(B), 0x4000, lib.BF16, 256, None, None) == lib.ERR_SHAPE
    B.cols = 256
    assert L.nvfp4_gemm(ctypes.byref(A), ctypes.byref(B), None, lib.BF16, 256, None, None) == lib.ERR_INVALID_ARG
    assert L.nvfp4_gemm(ctypes.byref(A), ctypes.byref(B), 0x4000, 9, 256, None, None) == lib.ERR_INVALID_ARG
    assert L.nvfp4_gemm(ctypes.byref(A), ctypes.byref(B), 0x4000, lib.BF16, 100, None, None) == lib.ERR_SHAPE
    A.cols = B.cols = 48                                                      # K % 32
    assert L.nvfp4_gemm(ctypes.byref(A), ctypes.byref(B), 0x4000, lib.BF16, 256, None, None) == lib.ERR_SHAPE
    A.cols = B.cols = 256
    A.codes = 0x1004
    assert L.nvfp4_gemm(ctypes.byref(A), ctypes.byref(B), 0x4000, lib.BF16, 256, None, None) == lib.ERR_ALIGNMENT
    W = lib.QTensorC(0x1000, None, 0x1000, 0x2000, None, None, 256, 256)
    assert L.nvfp4_linear_dgrad(0x1000, lib.BF16, 64, 256, 256, ctypes.byref(W), 0, 0, 0x4000, lib.BF16, 256,
                                0x8000, 1 << 30, None, None) == lib.ERR_INVALID_ARG   # no W^T copy
    assert L.nvfp4_linear_fprop(0x1000, lib.BF16, 64, 256, 256, ctypes.byref(W), 0x4000, lib.BF16, 256,
                                0x8000, 16, None, None) == lib.ERR_WORKSPACE
    assert L.nvfp4_selftest_wait_timeout(0, 0x1000, None) == lib.ERR_INVALID_ARG
    assert L.nvfp4_status_query(None, None) == lib.ERR_INVALID_ARG


def test_product_path_has_no_fallback(monkeypatch, lib):
    """With the library missing, the binding raises instead of computing elsewhere."""
    from nvfp4_bit_quantized_gb300 import _lib as L
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "LIB_PATH", "/nonexistent/libnvfp4_gb300.so")
    with pytest.raises(ImportError):
        L.lib()


@pytest.mark.parametrize("M,N,K", [(288, 416, 352), (8192, 20480, 5120), (16384, 14336, 4096), (32, 32, 32),
                                   (100, 3000, 64), (4096, 96, 5000)])
def test_linear_workspace_covers_every_operand_orientation(lib, M, N, K):
    """The linear workspace holds the amax partials plus slot A (X [M,K], dY [M,N] or
    dY^T [N,M]) and slot B (X^T [K,M]); tile-layout scale padding depends on the
    orientation, so each must fit."""
    L = lib.lib()

    def up16(v):
        return (v + 15) // 16 * 16

    def slot(r, c):
        return up16(r * c // 2) + up16(L.nvfp4_scales_mma_bytes(r, c)) + 16

    need = 4096 * 4 + max(slot(M, K), slot(M, N), slot(N, M)) + slot(K, M)
    assert L.nvfp4_linear_workspace_bytes(M, N, K) >= need


def test_mx_entry_points_reject_bad_arguments(lib):
    L = lib.lib()
    assert L.nvfp4_mx_scales_mma_bytes(128, 256) == 1024
    assert L.nvfp4_mx_scales_mma_bytes(129, 288) == 4096
    assert L.nvfp4_mx_scales_mma_bytes(8192, 5120) == 64 * 20 * 1024
    q = lib.QTensorC(0x1000, 0x1000, None, None, None, None, 32, 64)
    mxq = L.nvfp4_mx_quantize
    assert mxq(0x1000, 5, 32, 64, 64, 0, ctypes.byref(q), None) == lib.ERR_INVALID_ARG      # dtype
    assert mxq(0x1000, lib.BF16, 32, 64, 64, 2, ctypes.byref(q), None) == lib.ERR_INVALID_ARG  # col flag
    assert mxq(0x1000, lib.BF16, 32, 64, 48, 0, ctypes.byref(q), None) == lib.ERR_SHAPE     # ldx < C
    assert mxq(0x1000, lib.BF16, 32, 64, 64, 1, ctypes.byref(q), None) == lib.ERR_SHAPE     # x^T is [64, 32]
    q48 = lib.QTensorC(0x1000, 0x1000, None, None, None, None, 32, 48)
    assert mxq(0x1000, lib.BF16, 32, 48, 48, 0, ctypes.byref(q48), None) == lib.ERR_SHAPE   # 32-element blocks
    assert mxq(0x1010, lib.BF16, 32, 64, 64, 0, ctypes.byref(q), None) == lib.ERR_ALIGNMENT  # 32-byte loads
    assert mxq(0x1000, lib.BF16, 32, 64, 64, 0, None, None) == lib.ERR_INVALID_ARG
    big = 65536 * 64 + 32                                                    # x^T rows past the col grid
    qt = lib.QTensorC(0x1000, 0x1000, None, None, None, None, 64, big)
    assert mxq(0x1000, lib.BF16, big, 64, 64, 1, ctypes.byref(qt), None) == lib.ERR_SHAPE
    A = lib.QTensorC(0x1000, None, 0x1000, None, None, None, 128, 256)
    B = lib.QTensorC(0x1000, None, 0x1000, None, None, None, 256, 256)
    g = L.nvfp4_mx_gemm
    assert g(ctypes.byref(A), ctypes.byref(B), 0x4000, lib.F32, 256, None, None) == lib.ERR_UNSUPPORTED
    assert g(ctypes.byref(A), ctypes.byref(B), 0x4000, 9, 256, None, None) == lib.ERR_INVALID_ARG
    assert g(ctypes.byref(A), ctypes.byref(B), 0x4008, lib.BF16, 256, None, None) == lib.ERR_ALIGNMENT
    assert g(ctypes.byref(A), ctypes.byref(B), 0x4000, lib.BF16, 260, None, None) == lib.ERR_ALIGNMENT
    B.cols = 128
    assert g(ctypes.byref(A), ctypes.byref(B), 0x4000, lib.BF16, 256, None, None) == lib.ERR_SHAPE
    B.cols = 256
    B.scales_mma = None
    assert g(ctypes.byref(A), ctypes.byref(B), 0x4000, lib.BF16, 256, None, None) == lib.ERR_INVALID_ARG


def test_gemm_sqrelu_backward_rejects_bad_arguments(lib):
    L = lib.lib()
    A = lib.QTensorC(0x1000, None, 0x1000, 0x2000, None, None, 128, 256)
    B = lib.QTensorC(0x1000, None, 0x1000, 0x2000, None, None, 256, 256)
    f = L.nvfp4_gemm_sqrelu_bwd
    assert f(ctypes.byref(A), ctypes.byref(B), None, 256, 0x4000, 256, None, None) == lib.ERR_INVALID_ARG   # no H
    assert f(ctypes.byref(A), ctypes.byref(B), 0x8000, 200, 0x4000, 256, None, None) == lib.ERR_SHAPE       # ldh < N
    assert f(ctypes.byref(A), ctypes.byref(B), 0x8008, 256, 0x4000, 256, None, None) == lib.ERR_ALIGNMENT
    assert f(ctypes.byref(A), ctypes.byref(B), 0x8000, 260, 0x4000, 256, None, None) == lib.ERR_ALIGNMENT
    A.s_dec = None
    assert f(ctypes.byref(A), ctypes.byref(B), 0x8000, 256, 0x4000, 256, None, None) == lib.ERR_INVALID_ARG


def test_gemm_ws_rejects_bad_arguments_before_touching_the_device(lib):
    """nvfp4_gemm_ws: the shape and pointer checks of nvfp4_gemm come first (no device
    here); the workspace is sized per device, so without one the size is 0."""
    L = lib.lib()
    assert L.nvfp4_gemm_workspace_bytes(0) == 0 and L.nvfp4_gemm_workspace_bytes(-1) == 0
    A = lib.QTensorC(0x1000, None, 0x1000, 0x2000, None, None, 128, 256)
    B = lib.QTensorC(0x1000, None, 0x1000, 0x2000, None, None, 256, 128)     # K mismatch
    g = L.nvfp4_gemm_ws
    assert g(ctypes.byref(A), ctypes.byref(B), 0x4000, lib.BF16, 256, 0x8000, 1 << 20, None, None) == lib.ERR_SHAPE
    B.cols = 256
    assert g(ctypes.byref(A), ctypes.byref(B), None, lib.BF16, 256, 0x8000, 1 << 20, None, None) == lib.ERR_INVALID_ARG
    A.codes = 0x1004
    assert g(ctypes.byref(A), ctypes.byref(B), 0x4000, lib.BF16, 256, None, 0, None, None) == lib.ERR_ALIGNMENT


def test_sqrelu_maxima_entries_reject_bad_arguments(lib):
    L = lib.lib()
    # sized from the device's multiprocessor count: no device here, so 0 (never a fixed cap)
    assert L.nvfp4_sqrelu_maxima_bytes(0) == 0 and L.nvfp4_sqrelu_maxima_bytes(-1) == 0
    mb = 2 * 4 * 152 * 4
    A = lib.QTensorC(0x1000, None, 0x1000, 0x2000, None, None, 128, 256)
    B = lib.QTensorC(0x1000, None, 0x1000, 0x2000, None, None, 256, 256)
    f = L.nvfp4_gemm_sqrelu_maxima
    assert f(ctypes.byref(A), ctypes.byref(B), 0x4000, 256, 0, None, mb, None, None) == lib.ERR_INVALID_ARG   # no maxima
    assert f(ctypes.byref(A), ctypes.byref(B), 0x4000, 256, 0, 0x8002, mb, None, None) == lib.ERR_ALIGNMENT
    B.rows = 200                                                                                     # N % 16
    assert f(ctypes.byref(A), ctypes.byref(B), 0x4000, 256, 0, 0x8000, mb, None, None) == lib.ERR_SHAPE
    pr, pc = _qp(lib, 0, 0, 0), _qp(lib, 1, 0, 1)
    sdec = 0x2000
    qr = lib.QTensorC(0x1000, 0x1000, None, sdec, None, None, 32, 64)
    qc = lib.QTensorC(0x1000, 0x1000, None, sdec, None, None, 64, 32)
    q = L.nvfp4_quantize_dual_sqrelu_premax
    assert q(0x1000, lib.F32, 32, 64, 64, ctypes.byref(pr), ctypes.byref(qr), ctypes.byref(pc), ctypes.byref(qc),
             0x8000, mb, None, None) == lib.ERR_UNSUPPORTED
    assert q(0x1000, lib.BF16, 32, 64, 64, ctypes.byref(pr), ctypes.byref(qr), ctypes.byref(pc), ctypes.byref(qc),
             None, mb, None, None) == lib.ERR_INVALID_ARG
    assert q(0x1000, lib.BF16, 32, 64, 64, ctypes.byref(pc), ctypes.byref(qr), ctypes.byref(pc), ctypes.byref(qc),
             0x8000, mb, None, None) == lib.ERR_INVALID_ARG                                             # row params
    assert q(0x1000, lib.BF16, 32, 64, 64, ctypes.byref(pr), ctypes.byref(qr), ctypes.byref(pc), ctypes.byref(qc),
             0x8000, 4, None, None) == lib.ERR_WORKSPACE                                                # no partials


def test_dh_maxima_entries_reject_bad_arguments(lib):
    L = lib.lib()
    A = lib.QTensorC(0x1000, None, 0x1000, 0x2000, None, None, 128, 256)
    B = lib.QTensorC(0x1000, None, 0x1000, 0x2000, None, None, 256, 256)
    f = L.nvfp4_gemm_sqrelu_bwd_maxima
    mb = 2 * 4 * 152 * 4
    assert f(ctypes.byref(A), ctypes.byref(B), 0x8000, 256, 0x4000, 256, 0, None, mb, None, None) == lib.ERR_INVALID_ARG
    assert f(ctypes.byref(A), ctypes.byref(B), 0x8000, 256, 0x4000, 256, 0, 0x9002, mb, None, None) == lib.ERR_ALIGNMENT
    B.rows = 200                                                                                     # N % 16
    assert f(ctypes.byref(A), ctypes.byref(B), 0x8000, 256, 0x4000, 256, 0, 0x9000, mb, None, None) == lib.ERR_SHAPE
    pr, pc = _qp(lib, 0, 1, 0), _qp(lib, 1, 1, 1)
    qr = lib.QTensorC(0x1000, 0x1000, None, 0x2000, None, None, 32, 64)
    qc = lib.QTensorC(0x1000, 0x1000, None, 0x2000, None, None, 64, 32)
    q = L.nvfp4_quantize_dual_premax
    assert q(0x1000, lib.F32, 32, 64, 64, ctypes.byref(pr), ctypes.byref(qr), ctypes.byref(pc), ctypes.byref(qc),
             0x8000, mb, None, None) == lib.ERR_UNSUPPORTED
    assert q(0x1000, lib.BF16, 32, 64, 64, ctypes.byref(pr), ctypes.byref(qr), ctypes.byref(pc), ctypes.byref(qc),
             None, mb, None, None) == lib.ERR_INVALID_ARG
