"""Guard canaries: every output buffer of the C ABI is surrounded by 4 KB of a fill
pattern, and after each call (ragged shapes, every kernel family) the pattern must be
intact -- no kernel writes outside the buffers it was given.  Stands in for a memory
checker, which this GPU pool does not offer."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu
G = 4096
FILL = 0xA5


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_bit_quantized_gb300 as nv
    return nv


class Guarded:
    """Device buffers of `nbytes` with G guard bytes on each side, all filled with FILL."""

    def __init__(self):
        self.bufs = []

    def __call__(self, nbytes: int) -> int:
        t = torch.full((max(nbytes, 1) + 2 * G,), FILL, dtype=torch.uint8, device="cuda")
        self.bufs.append((t, max(nbytes, 1)))
        return t.data_ptr() + G

    def check(self):
        torch.cuda.synchronize()
        for t, n in self.bufs:
            assert bool((t[:G] == FILL).all()) and bool((t[G + n:] == FILL).all()), "write outside a buffer"


def _x(R, C, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((R, C), generator=g) * 2).to(dtype).cuda()


def _qt(L, gb, rows, cols, block=0, transpose=False, mx=False):
    lib = L.lib()
    smma = int(lib.nvfp4_mx_scales_mma_bytes(rows, cols) if mx else lib.nvfp4_scales_mma_bytes(rows, cols))
    sc = rows * cols // (32 if mx else 16) if block != 2 else (rows // 16) * (cols // 16)
    q = L.QTensorC(gb(rows * cols // 2), gb(sc), gb(smma), None if mx else gb(16), None, None, rows, cols)
    if transpose:
        q.codes_t = gb(rows * cols // 2)
        q.scales_mma_t = gb(int(lib.nvfp4_scales_mma_bytes(cols, rows)))
    return q


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("R,C", [(208, 336), (64, 1056), (1, 32)])
def test_quantizers_stay_inside_their_buffers(nv, dtype, R, C):
    from nvfp4_bit_quantized_gb300 import _lib as L
    lib, gb = L.lib(), Guarded()
    x = _x(R, C, dtype, R + C)
    st = nv.dev_status().data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    dt = L.F32 if dtype == torch.float32 else L.BF16
    ws = gb(1 << 20)
    modes = [(L.ROW, L.RNE, 0), (L.ROW, L.SR, 0)]
    if R % 16 == 0:
        modes += [(L.COL, L.SR, 1), (L.COL, L.RNE, 0), (L.TILE16, L.RNE, 0)]
    for block, rnd, rht in modes:
        rows, cols = (C, R) if block == L.COL else (R, C)
        q = _qt(L, gb, rows, cols, block, transpose=block == L.TILE16)
        p = L.QParams(block, rnd, rht, 1, 3, 5)
        assert lib.nvfp4_quantize(x.data_ptr(), dt, R, C, C, ctypes.byref(p), ctypes.byref(q), ws, 1 << 20, st, s) == 0
    if R % 16 == 0:
        qr, qc = _qt(L, gb, R, C), _qt(L, gb, C, R)
        pr, pc = L.QParams(L.ROW, L.SR, 0, 1, 3, 5), L.QParams(L.COL, L.SR, 1, 1, 3, 5)
        assert lib.nvfp4_quantize_dual(x.data_ptr(), dt, R, C, C, ctypes.byref(pr), ctypes.byref(qr), ctypes.byref(pc),
                                       ctypes.byref(qc), ws, 1 << 20, st, s) == 0
    if C % 32 == 0:
        assert lib.nvfp4_mx_quantize(x.data_ptr(), dt, R, C, C, 0, ctypes.byref(_qt(L, gb, R, C, mx=True)), s) == 0
    if R % 32 == 0:
        assert lib.nvfp4_mx_quantize(x.data_ptr(), dt, R, C, C, 1, ctypes.byref(_qt(L, gb, C, R, mx=True)), s) == 0
    gb.check()
    assert nv.status_query() == 0


@pytest.mark.parametrize("M,N,K", [(200, 296, 224), (400, 528, 1056), (16, 16, 32)])
def test_gemms_stay_inside_their_buffers(nv, M, N, K):
    from nvfp4_bit_quantized_gb300 import _lib as L
    lib, gb = L.lib(), Guarded()
    st = nv.dev_status().data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    qa = nv.quantize(_x(M, K, torch.bfloat16, 1), nv.ROW, nv.RNE)
    qb = nv.quantize(_x(N, K, torch.bfloat16, 2) * 0.02, nv.ROW, nv.RNE)
    a, b = qa.c_struct(), qb.c_struct()
    for path in (1, 2):
        lib.nvfp4_gemm_force_path(path)
        try:
            for dt, esz in ((L.BF16, 2), (L.F32, 4)):
                assert lib.nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), gb(M * N * esz), dt, N, st, s) == 0
        finally:
            lib.nvfp4_gemm_force_path(0)
    H = _x(M, N, torch.bfloat16, 3)
    assert lib.nvfp4_gemm_sqrelu_bwd(ctypes.byref(a), ctypes.byref(b), H.data_ptr(), N, gb(M * N * 2), N, st, s) == 0
    mbytes = int(lib.nvfp4_sqrelu_maxima_bytes(torch.cuda.current_device()))
    if M % 16 == 0 and N % 16 == 0:
        assert lib.nvfp4_gemm_sqrelu_bwd_maxima(ctypes.byref(a), ctypes.byref(b), H.data_ptr(), N, gb(M * N * 2), N,
                                                7, gb(mbytes), mbytes, st, s) == 0
        assert lib.nvfp4_gemm_sqrelu_maxima(ctypes.byref(a), ctypes.byref(b), gb(M * N * 2), N, 7, gb(mbytes),
                                            mbytes, st, s) == 0
    ma = nv.mx_quantize(_x(M, K, torch.bfloat16, 4))
    mb = nv.mx_quantize(_x(N, K, torch.bfloat16, 5))
    mac, mbc = ma.c_struct(), mb.c_struct()
    assert lib.nvfp4_mx_gemm(ctypes.byref(mac), ctypes.byref(mbc), gb(M * N * 2), L.BF16, N, st, s) == 0
    gb.check()
    assert nv.status_query() == 0
