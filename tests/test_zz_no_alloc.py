"""The allocation-free quantize entry point, through the C ABI.

nvfp4_quantize_noalloc serves callers that can pass their inputs and outputs
but cannot obtain an extra device buffer for the workspace nvfp4_quantize asks
for (its scratch lives in a static device array inside the library).  Its
results must equal nvfp4_quantize's bit for bit -- the tolerance every
quantizer test here uses -- on two calls in a row (the second call reuses the
array the first one left behind).  This file is collected last and passes
both alone and after the other tests.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

CASES = [  # (block, round, rht, shape, dtype)
    (0, 0, 0, (300, 512), torch.bfloat16),
    (0, 1, 0, (64, 5120), torch.bfloat16),
    (1, 1, 1, (256, 336), torch.bfloat16),
    (1, 0, 1, (128, 64), torch.float32),
    (2, 0, 0, (208, 352), torch.bfloat16),
]


def _alloc(rows, cols, block, dev):
    from nvfp4_bit_quantized_gb300 import api
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty((rows // 16, cols // 16) if block == 2 else (rows, cols // 16), dtype=torch.uint8, device=dev)
    smma = torch.empty(max(api.scales_mma_bytes(rows, cols), 16), dtype=torch.uint8, device=dev)
    s_dec = torch.empty(4, dtype=torch.float32, device=dev)
    return codes, scales, smma, s_dec


@pytest.mark.parametrize("block,rnd,rht,shape,dtype", CASES)
def test_noalloc_matches_workspace_entry_point(block, rnd, rht, shape, dtype):
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_bit_quantized_gb300 as nv
    from nvfp4_bit_quantized_gb300 import _lib as L

    lib = L.lib()
    dev = torch.device("cuda", 0)
    g = torch.Generator(device="cpu").manual_seed(hash((block, rnd, shape)) % 10007)
    R, C = shape
    rows, cols = (C, R) if block == 1 else (R, C)
    params = L.QParams(block, rnd, rht, 3, 1234, 77)
    stream = torch.cuda.current_stream().cuda_stream
    nv.reset_status()
    for call in range(2):
        x = (torch.randn(shape, generator=g) * (1e-3 if rnd else 1.0)).to(dtype).to(dev)
        ref = nv.quantize(x, block, rnd, rht=bool(rht), sr_seed=1234, sr_offset=3, rht_seed=77, transpose=False)
        codes, scales, smma, s_dec = _alloc(rows, cols, block, dev)
        q = L.QTensorC(codes.data_ptr(), scales.data_ptr(), smma.data_ptr(), s_dec.data_ptr(), None, None, rows, cols)
        st = lib.nvfp4_quantize_noalloc(x.data_ptr(), L.BF16 if dtype == torch.bfloat16 else L.F32, R, C,
                                        x.stride(0), ctypes.byref(params), ctypes.byref(q),
                                        nv.dev_status().data_ptr(), stream)
        assert st == L.OK, L.status_string(st)
        assert nv.status_query() == 0
        assert torch.equal(codes, ref.codes), f"call {call}: codes differ"
        assert torch.equal(scales, ref.scales), f"call {call}: scales differ"
        assert torch.equal(smma[:ref.scales_mma.numel()], ref.scales_mma), f"call {call}: tile scales differ"
        assert torch.equal(s_dec[:1], ref.s_dec[:1]), f"call {call}: s_dec differs"


def test_noalloc_rejects_bad_arguments_like_the_workspace_entry_point():
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_bit_quantized_gb300 import _lib as L
    lib = L.lib()
    params = L.QParams(7, 0, 0, 0, 0, 0)            # bad block
    q = L.QTensorC(0x1000, 0x1000, None, 0x2000, None, None, 32, 64)
    assert lib.nvfp4_quantize_noalloc(0x1000, L.BF16, 32, 64, 64, ctypes.byref(params), ctypes.byref(q),
                                      None, None) == L.ERR_INVALID_ARG
    assert lib.nvfp4_quantize_noalloc(0x1000, L.BF16, 32, 64, 64, None, ctypes.byref(q), None, None) == \
        L.ERR_INVALID_ARG
