"""MXFP4, the comparison format: the GPU quantizer bit for bit against the oracle
(codes, UE8M0 scales, the tensor-core scale layout), the MXFP4 GEMM within 1e-3 of
the fp64 oracle GEMM on identical dequantized operands, and the format comparison
on heavy-tailed data (NVFP4's quantization error below MXFP4's)."""
import numpy as np
import pytest
import torch

from helpers import bf16_round, host_input, mx_mma_layout_from_canonical, rel_fro

pytestmark = pytest.mark.gpu
TOL = 1e-3


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_bit_quantized_gb300 as nv
    return nv


def _input(shape, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g) * torch.exp(torch.randn((shape[0], 1), generator=g) * 3)
    x = x.to(dtype)
    x.view(-1)[:8] = torch.tensor([0.0, -0.0, 1e-30, -1e-30, 2.5, -3.5, 5.0, 0.75], dtype=dtype)
    if shape[1] >= 64:
        x[0, 32:64] = 0                                          # an all-zero block
    return x


def _same(nv, q, ref):
    torch.cuda.synchronize()
    assert np.array_equal(q.codes.cpu().numpy(), ref["codes"])
    assert np.array_equal(q.scales.cpu().numpy(), ref["scales"])
    assert np.array_equal(q.scales_mma.cpu().numpy()[:nv.mx_scales_mma_bytes(q.rows, q.cols)],
                          mx_mma_layout_from_canonical(ref["scales"], q.rows, q.cols))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", [(1, 32), (200, 96), (256, 512), (96, 800), (130, 1056)])
def test_mx_quantize_rows_bit_exact(nv, oracle_mod, dtype, shape):
    x = _input(shape, dtype, seed=sum(shape))
    q = nv.mx_quantize(x.cuda())
    _same(nv, q, oracle_mod.mx_quantize(host_input(x)))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", [(32, 8), (96, 200), (512, 256), (800, 96), (1056, 136)])
def test_mx_quantize_cols_bit_exact(nv, oracle_mod, dtype, shape):
    x = _input(shape, dtype, seed=7 * sum(shape))
    q = nv.mx_quantize(x.cuda(), col=True)
    _same(nv, q, oracle_mod.mx_quantize(host_input(x), col=True))


def test_mx_quantize_strided_input(nv, oracle_mod):
    x = _input((64, 320), torch.bfloat16, seed=3)
    big = torch.zeros((64, 384), dtype=torch.bfloat16)
    big[:, :320] = x
    g = big.cuda()[:, :320]
    for col in (False, True):
        _same(nv, nv.mx_quantize(g, col=col), oracle_mod.mx_quantize(host_input(x), col=col))
    # x^T of a view whose column count (130) ends inside a 16-byte piece
    y = _input((96, 130), torch.bfloat16, seed=4)
    big = torch.zeros((96, 136), dtype=torch.bfloat16)
    big[:, :130] = y
    _same(nv, nv.mx_quantize(big.cuda()[:, :130], col=True), oracle_mod.mx_quantize(host_input(y), col=True))


def _mx_ref(oracle_mod, q):
    return dict(codes=q.codes.cpu().numpy(), scales=q.scales.cpu().numpy(), rows=q.rows, cols=q.cols)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (128, 256, 512), (300, 520, 352), (1000, 296, 224),
                                   (1, 8, 32), (2048, 2048, 2048)])
def test_mx_gemm_matches_oracle(nv, oracle_mod, M, N, K):
    g = torch.Generator().manual_seed(M + N + K)
    A = torch.randn((M, K), generator=g).to(torch.bfloat16).cuda()
    B = (torch.randn((N, K), generator=g) * 0.02).to(torch.bfloat16).cuda()
    qa, qb = nv.mx_quantize(A), nv.mx_quantize(B)
    nv.reset_status()
    D = nv.mx_gemm(qa, qb)
    assert nv.status_query() == 0
    ref = oracle_mod.gemm_f64(oracle_mod.mx_dequant(_mx_ref(oracle_mod, qa)),
                              oracle_mod.mx_dequant(_mx_ref(oracle_mod, qb)))
    assert rel_fro(D.float().cpu().numpy(), bf16_round(ref)) <= TOL


def test_mx_gemm_transposed_operands_and_wide_scale_range(nv, oracle_mod):
    """Wgrad-shaped product of two column operands, with rows spanning 2^-40 .. 2^40
    so the UE8M0 scales cover a wide range."""
    T, d, f = 512, 256, 384
    g = torch.Generator().manual_seed(5)
    dY = (torch.randn((T, f), generator=g) * torch.exp2(torch.randint(-40, 40, (T, 1), generator=g).float()))
    X = torch.randn((T, d), generator=g)
    qa = nv.mx_quantize(dY.to(torch.bfloat16).cuda(), col=True)      # dY^T [f, T]
    qb = nv.mx_quantize(X.to(torch.bfloat16).cuda(), col=True)       # X^T [d, T]
    D = nv.mx_gemm(qa, qb)
    ref = oracle_mod.gemm_f64(oracle_mod.mx_dequant(_mx_ref(oracle_mod, qa)),
                              oracle_mod.mx_dequant(_mx_ref(oracle_mod, qb)))
    assert rel_fro(D.float().cpu().numpy(), bf16_round(ref)) <= TOL


def test_mx_gemm_full_fprop_shape_sampled(nv, oracle_mod):
    """8192 x 5120 x 20480 (the FFN up-projection), sampled 64 x 64 output blocks."""
    from nvfp4_bit_quantized_gb300 import inputs
    M, K, N = 8192, 5120, 20480
    X = inputs.normal((M, K), 1.0, 20, device="cuda")
    W = inputs.normal((N, K), 0.02, 21, device="cuda")
    qa, qb = nv.mx_quantize(X), nv.mx_quantize(W)
    nv.reset_status()
    D = nv.mx_gemm(qa, qb)
    assert nv.status_query() == 0
    rng = np.random.default_rng(6)
    A, B = _mx_ref(oracle_mod, qa), _mx_ref(oracle_mod, qb)
    for m, n in ((0, 0), (M - 64, N - 64), (int(rng.integers(0, M // 64)) * 64, int(rng.integers(0, N // 64)) * 64)):
        ref = oracle_mod.gemm_f64(oracle_mod.mx_dequant(A, m, m + 64), oracle_mod.mx_dequant(B, n, n + 64))
        assert rel_fro(D[m:m + 64, n:n + 64].float().cpu().numpy(), bf16_round(ref)) <= TOL, (m, n)


def test_nvfp4_quantization_error_below_mxfp4_on_heavy_tailed_data(nv, oracle_mod):
    """The format comparison without training: on the heavy-tailed layer's activations
    (Student-t(3), 1% of channels x50) NVFP4's relative dequantization error is below
    MXFP4's, on the GPU's own codes and scales (dequantized by the oracle)."""
    from nvfp4_bit_quantized_gb300 import inputs
    X, _, _ = inputs.heavy_tailed_layer(512, 4096, 256, seed=3, device="cuda")
    xf = X.float().cpu().numpy().astype(np.float64)
    qn = nv.quantize(X, nv.ROW, nv.RNE)
    qm = nv.mx_quantize(X)
    dn = oracle_mod.dequant(dict(codes=qn.codes.cpu().numpy(), scales=qn.scales.cpu().numpy(),
                                 s_dec=float(qn.s_dec[0].item()), rows=qn.rows, cols=qn.cols, block=0))
    dm = oracle_mod.mx_dequant(_mx_ref(oracle_mod, qm))
    en, em = rel_fro(dn, xf), rel_fro(dm, xf)
    assert 0 < en < em, (en, em)
