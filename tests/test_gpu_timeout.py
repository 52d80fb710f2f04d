"""Bounded waits: a barrier nobody arrives at times out, the status says so,
and the context stays usable (no GPU fault, no hang)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_wait_timeout_sets_status_and_context_survives():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_bit_quantized_gb300 as nv
    from nvfp4_bit_quantized_gb300 import _lib as L
    nv.reset_status()
    st = L.lib().nvfp4_selftest_wait_timeout(20_000_000, nv.dev_status().data_ptr(),
                                              torch.cuda.current_stream().cuda_stream)
    assert st == 0
    assert nv.status_query() == L.ERR_TIMEOUT
    nv.reset_status()
    x = torch.randn((64, 64), device="cuda").to(torch.bfloat16)
    q = nv.quantize(x, nv.ROW)
    assert nv.status_query() == 0
    assert q.s_dec[0].item() > 0
