"""Programmatic dependent launch: every library kernel may start while its predecessor in the
stream drains and waits (griddepcontrol.wait) before touching global memory.  These tests
chain library kernels with each other, with torch kernels that write their inputs, and inside
a captured CUDA graph, and check the results against the oracle or against eager runs."""
import numpy as np
import pytest
import torch

from helpers import host_input

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_bit_quantized_gb300 as nv
    return nv


def test_quantize_sees_the_writes_of_the_torch_kernel_before_it(nv, oracle_mod):
    """A torch kernel rewrites x in place right before each quantization (no synchronisation
    in between): every quantization equals the oracle's of the values that kernel wrote."""
    g = torch.Generator(device="cpu").manual_seed(3)
    x = torch.randn((1024, 2048), generator=g).to(torch.bfloat16).cuda()
    outs, refs = [], []
    for i in range(4):
        x.mul_(-1.5 if i % 2 else 3.0)
        outs.append(nv.quantize(x, nv.ROW, nv.SR, sr_seed=i))
        refs.append(x.clone())
    torch.cuda.synchronize()
    for i, (q, xr) in enumerate(zip(outs, refs)):
        r = oracle_mod.quantize(host_input(xr), oracle_mod.ROW, oracle_mod.SR, sr_seed=i)
        assert np.array_equal(q.codes.cpu().numpy(), r["codes"]), i
        assert np.array_equal(q.scales.cpu().numpy(), r["scales"]), i


def _chain(nv, X, W):
    """Quantize -> GEMM -> quantize the GEMM's output -> GEMM: each step reads what the one
    before it wrote."""
    xq = nv.quantize(X, nv.ROW, nv.RNE, scales=False)
    wq = nv.quantize(W, nv.TILE16, nv.RNE, scales=False, transpose=True)
    H = nv.gemm(xq, wq, torch.bfloat16)
    hq, ht = nv.quantize_dual(H, nv.SR, nv.SR, rht=True, sr_seed=5, rht_seed=6, scales=False)
    D = nv.gemm(hq, wq.transposed(), torch.bfloat16, split_tail=True)
    return H, D, hq.codes, ht.codes


def test_kernel_chain_in_a_cuda_graph_equals_eager(nv):
    g = torch.Generator(device="cpu").manual_seed(4)
    X = torch.randn((2048, 1024), generator=g).to(torch.bfloat16).cuda()
    W = (torch.randn((2560, 1024), generator=g) * 0.02).to(torch.bfloat16).cuda()
    nv.reset_status()
    eager = [t.clone() for t in _chain(nv, X, W)]
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    _chain(nv, X, W)                              # warm-up on the capture stream's allocator
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        captured = _chain(nv, X, W)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert nv.status_query() == 0
    for a, b in zip(eager, captured):
        assert torch.equal(a, b)


def test_back_to_back_gemms_into_one_output_in_order(nv):
    """Two GEMMs write the same output in a row and a third reads it as its input: the last
    writer wins and the reader sees it (no reordering between dependent launches)."""
    g = torch.Generator(device="cpu").manual_seed(5)
    A = torch.randn((1024, 512), generator=g).to(torch.bfloat16).cuda()
    B1 = (torch.randn((768, 512), generator=g) * 0.02).to(torch.bfloat16).cuda()
    B2 = (torch.randn((768, 512), generator=g) * 0.05).to(torch.bfloat16).cuda()
    aq = nv.quantize(A, nv.ROW, nv.RNE)
    b1, b2 = nv.quantize(B1, nv.ROW, nv.RNE), nv.quantize(B2, nv.ROW, nv.RNE)
    out = torch.empty((1024, 768), dtype=torch.bfloat16, device="cuda")
    nv.gemm(aq, b1, out=out)
    nv.gemm(aq, b2, out=out)
    q_after = nv.quantize(out, nv.ROW, nv.RNE)
    expect = nv.gemm(aq, b2, torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(out, expect)
    q_ref = nv.quantize(expect, nv.ROW, nv.RNE)
    torch.cuda.synchronize()
    assert torch.equal(q_after.codes, q_ref.codes) and torch.equal(q_after.scales, q_ref.scales)
