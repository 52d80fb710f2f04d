"""The three linear-layer entry points against the oracle end to end: the
oracle quantizes the same inputs itself (bit-exact with the GPU, so the
dequantized operands are identical) and runs the fp64 GEMM."""
import numpy as np
import pytest
import torch

from helpers import bf16_round, host_input, rel_fro

pytestmark = pytest.mark.gpu
TOL = 1e-3


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_bit_quantized_gb300 as nv
    return nv


def _layer_refs(oracle_mod, X, W, dY, sr_seed, rht_seed):
    x, w, dy = host_input(X), host_input(W), host_input(dY)
    rx = oracle_mod.quantize(x, oracle_mod.ROW)
    rw = oracle_mod.quantize(w, oracle_mod.TILE16)
    rwt = oracle_mod.quantize(np.ascontiguousarray(w.T), oracle_mod.TILE16)
    rdy = oracle_mod.quantize(dy, oracle_mod.ROW, oracle_mod.SR, sr_seed=sr_seed)
    rdyt = oracle_mod.quantize(dy, oracle_mod.COL, oracle_mod.SR, rht=True, sr_seed=sr_seed, rht_seed=rht_seed)
    rxt = oracle_mod.quantize(x, oracle_mod.COL, oracle_mod.RNE, rht=True, rht_seed=rht_seed)
    deq = oracle_mod.dequant
    Y = oracle_mod.gemm_f64(deq(rx), deq(rw))
    dX = oracle_mod.gemm_f64(deq(rdy), deq(rwt))
    dW = oracle_mod.gemm_f64(deq(rdyt), deq(rxt))
    return Y, dX, dW


def test_single_layer_fp32_config(nv, oracle_mod):
    """The small single-layer case: M = K = N = 256, fp32 inputs and outputs, seed 0,
    SR Philox seed 0, RHT sign seed 1."""
    from nvfp4_bit_quantized_gb300 import inputs
    X, W, dY = inputs.linear_layer(256, 256, 256, seed=0, dtype=torch.float32, device="cpu")
    Xg, Wg, dYg = X.cuda(), W.cuda(), dY.cuda()
    nv.reset_status()
    wq = nv.quantize_weight(Wg)
    Y = nv.linear_fprop(Xg, wq, torch.float32)
    dX = nv.linear_dgrad(dYg, wq, sr_seed=0, out_dtype=torch.float32)
    dW = nv.linear_wgrad(dYg, Xg, sr_seed=0, rht_seed=1, out_dtype=torch.float32)
    assert nv.status_query() == 0
    rY, rdX, rdW = _layer_refs(oracle_mod, Xg, Wg, dYg, 0, 1)
    for got, ref in ((Y, rY), (dX, rdX), (dW, rdW)):
        assert rel_fro(got.cpu().numpy(), ref) <= TOL


def test_layer_bf16_ragged(nv, oracle_mod):
    """bf16 in/out, M = 288, K = 352, N = 416: none a tile multiple (each GEMM's
    contraction length must be a multiple of 32)."""
    from nvfp4_bit_quantized_gb300 import inputs
    X, W, dY = inputs.linear_layer(288, 352, 416, seed=3, dtype=torch.bfloat16, device="cpu")
    Xg, Wg, dYg = X.cuda(), W.cuda(), dY.cuda()
    wq = nv.quantize_weight(Wg)
    Y = nv.linear_fprop(Xg, wq)
    dX = nv.linear_dgrad(dYg, wq, sr_seed=11, sr_offset=2)
    dW = nv.linear_wgrad(dYg, Xg, sr_seed=11, sr_offset=2, rht_seed=5)
    torch.cuda.synchronize()
    x, w, dy = host_input(Xg), host_input(Wg), host_input(dYg)
    rY, _, _ = _layer_refs(oracle_mod, Xg, Wg, dYg, 11, 5)
    assert rel_fro(Y.float().cpu().numpy(), bf16_round(rY)) <= TOL
    rdy = oracle_mod.quantize(dy, oracle_mod.ROW, oracle_mod.SR, sr_seed=11, sr_offset=2)
    rwt = oracle_mod.quantize(np.ascontiguousarray(w.T), oracle_mod.TILE16)
    rdX = oracle_mod.gemm_f64(oracle_mod.dequant(rdy), oracle_mod.dequant(rwt))
    assert rel_fro(dX.float().cpu().numpy(), bf16_round(rdX)) <= TOL
    rdyt = oracle_mod.quantize(dy, oracle_mod.COL, oracle_mod.SR, rht=True, sr_seed=11, sr_offset=2, rht_seed=5)
    rxt = oracle_mod.quantize(x, oracle_mod.COL, oracle_mod.RNE, rht=True, rht_seed=5)
    rdW = oracle_mod.gemm_f64(oracle_mod.dequant(rdyt), oracle_mod.dequant(rxt))
    assert rel_fro(dW.float().cpu().numpy(), bf16_round(rdW)) <= TOL


def test_wgrad_rht_preserves_product(nv):
    """(R dY)^T (R X) = dY^T X: the RHT Wgrad is close to the plain product."""
    M, N, K = 1024, 256, 256
    g = torch.Generator(device="cpu").manual_seed(21)
    X = torch.randn((M, K), generator=g).to(torch.bfloat16).cuda()
    dY = (torch.randn((M, N), generator=g) * 1e-3).to(torch.bfloat16).cuda()
    dW = nv.linear_wgrad(dY, X, sr_seed=1, rht_seed=2, out_dtype=torch.float32)
    exact = dY.double().t() @ X.double()
    err = (dW.double() - exact).norm() / exact.norm()
    assert err < 0.2, float(err)      # 4-bit quantization noise, not a parity bound
