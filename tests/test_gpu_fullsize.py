"""Parity at the full workload sizes, in the launch configuration bench.py times.

The oracle cannot run a whole 8192 x 5120 x 20480 layer in test time, so it
checks samples: every quantized operand bit for bit on sampled row ranges (the
oracle still takes the tensor amax over the whole tensor, RHT included), and
every GEMM on sampled output blocks -- including the last, ragged-free edge
block -- against its fp64 product of the GPU's own codes and scales.
"""
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


def _mma_rows(buf: np.ndarray, rows, cols: int, tile2d: bool = False):
    """Scale bytes of the given operand rows, read back from the tensor-core layout."""
    nkb = (cols + 255) // 256
    r = np.asarray(rows)[:, None]
    s = np.arange(cols // 16)[None, :]
    off = (((r >> 7) * nkb + (s >> 4)) << 11) + (((s >> 2) & 3) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (s & 3)
    return buf[off]


def _check_operand(oracle_mod, q, x_host, block, rnd, rht, sr_seed, sr_offset, rht_seed, starts, n=16):
    """Bit-exact comparison of a GPU-quantized operand with the oracle on row ranges."""
    codes = q.codes.cpu().numpy()
    scales = q.scales.cpu().numpy()
    smma = q.scales_mma.cpu().numpy()
    for r0 in starts:
        r0 = int(r0) - int(r0) % 16
        r1 = min(r0 + n, q.rows)
        ref = oracle_mod.quantize(x_host, block, rnd, rht=rht, sr_seed=sr_seed, sr_offset=sr_offset,
                                  rht_seed=rht_seed, row_begin=r0, row_end=r1)
        assert np.float32(q.s_dec[0].item()) == np.float32(ref["s_dec"])
        assert np.array_equal(codes[r0:r1], ref["codes"][r0:r1]), (block, r0)
        if block == oracle_mod.TILE16:
            assert np.array_equal(scales[r0 // 16:r1 // 16], ref["scales"][r0 // 16:r1 // 16])
            exp = np.repeat(ref["scales"][r0 // 16:r1 // 16], 16, axis=0)
        else:
            assert np.array_equal(scales[r0:r1], ref["scales"][r0:r1]), (block, r0)
            exp = ref["scales"][r0:r1]
        assert np.array_equal(_mma_rows(smma, np.arange(r0, r1), q.cols), exp)


def _gemm_blocks(oracle_mod, qa, qb, D, blocks, a_tile=False, b_tile=False):
    """GPU output blocks vs the fp64 oracle product of the GPU codes and scales."""
    def deq(q, tile, rows):
        d = dict(codes=q.codes.cpu().numpy(), scales=q.scales.cpu().numpy(), s_dec=float(q.s_dec[0].item()),
                 rows=q.rows, cols=q.cols, block=oracle_mod.TILE16 if tile else oracle_mod.ROW)
        return oracle_mod.dequant(d, rows[0], rows[1])
    Dh = D.float().cpu().numpy()
    for (m0, m1), (n0, n1) in blocks:
        ref = oracle_mod.gemm_f64(deq(qa, a_tile, (m0, m1)), deq(qb, b_tile, (n0, n1)))
        err = rel_fro(Dh[m0:m1, n0:n1], bf16_round(ref))
        assert err <= TOL, ((m0, n0), err)


def _blocks(M, N, rng, n=3, size=64):
    out = [((0, size), (0, size)), ((M - size, M), (N - size, N))]
    for _ in range(n):
        m = int(rng.integers(0, M // size)) * size
        k = int(rng.integers(0, N // size)) * size
        out.append(((m, m + size), (k, k + size)))
    return out


def _layer(nv, oracle_mod, X, W, dY, seed):
    """The bench step's quantizations and GEMMs (bf16 out), checked on samples."""
    rng = np.random.default_rng(seed)
    M, K = X.shape
    N = W.shape[0]
    wq = nv.quantize(W, nv.TILE16, nv.RNE, transpose=True)
    xq = nv.quantize(X, nv.ROW, nv.RNE)
    dyq = nv.quantize(dY, nv.ROW, nv.SR, sr_seed=7, sr_offset=3)
    dyt = nv.quantize(dY, nv.COL, nv.SR, rht=True, sr_seed=7, sr_offset=3, rht_seed=11)
    xt = nv.quantize(X, nv.COL, nv.RNE, rht=True, rht_seed=11)
    # the bench's dual quantizations (one read of X / dY for both operands) equal the single calls
    dxr, dxc = nv.quantize_dual(X, nv.RNE, nv.RNE, rht=True, rht_seed=11)
    dyr, dyc = nv.quantize_dual(dY, nv.SR, nv.SR, rht=True, sr_seed=7, sr_offset=3, rht_seed=11)
    for d, s in ((dxr, xq), (dxc, xt), (dyr, dyq), (dyc, dyt)):
        assert torch.equal(d.codes, s.codes) and torch.equal(d.scales, s.scales)
        assert torch.equal(d.scales_mma, s.scales_mma) and torch.equal(d.s_dec[:1], s.s_dec[:1])
    del dxr, dxc, dyr, dyc
    nv.reset_status()
    Y = nv.gemm(xq, wq, torch.bfloat16)
    dX = nv.gemm(dyq, wq.transposed(), torch.bfloat16)
    dW = nv.gemm(dyt, xt, torch.bfloat16)
    assert nv.status_query() == 0
    x, w, dy = host_input(X), host_input(W), host_input(dY)
    o = oracle_mod
    _check_operand(o, xq, x, o.ROW, o.RNE, False, 0, 0, 0, [0, rng.integers(0, M), M - 16])
    _check_operand(o, wq, w, o.TILE16, o.RNE, False, 0, 0, 0, [0, rng.integers(0, N), N - 16])
    _check_operand(o, dyq, dy, o.ROW, o.SR, False, 7, 3, 0, [0, rng.integers(0, M), M - 16])
    _check_operand(o, dyt, dy, o.COL, o.SR, True, 7, 3, 11, [0, rng.integers(0, N), N - 16])
    _check_operand(o, xt, x, o.COL, o.RNE, True, 0, 0, 11, [0, rng.integers(0, K), K - 16])
    # W^T copy: its rows are W's columns
    wt_ref = o.quantize(np.ascontiguousarray(w[:, :]).T.copy(), o.TILE16, row_begin=0, row_end=32)
    assert np.array_equal(wq.codes_t.cpu().numpy()[:32], wt_ref["codes"][:32])
    wtq = wq.transposed()
    wtq_full = type(wtq)(wq.codes_t, wq.scales.t().contiguous(), wq.scales_mma_t, wq.s_dec, K, N, nv.TILE16)
    _gemm_blocks(o, xq, wq, Y, _blocks(M, N, rng), b_tile=True)
    _gemm_blocks(o, dyq, wtq_full, dX, _blocks(M, K, rng), b_tile=True)
    _gemm_blocks(o, dyt, xt, dW, _blocks(N, K, rng))


def test_ffn_up_projection_full_size(nv, oracle_mod):
    """M = 8192, K = 5120, N = 20480, bf16: the bench workload."""
    from nvfp4_bit_quantized_gb300 import inputs
    X, W, dY = inputs.linear_layer(8192, 5120, 20480, seed=0, dtype=torch.bfloat16, device="cuda")
    _layer(nv, oracle_mod, X, W, dY, seed=1)


def test_heavy_tailed_layer_full_size(nv, oracle_mod):
    """M = 16384, K = 4096, N = 14336: Student-t(3) activations with 1% of channels
    x50, Student-t(4) x 1e-3 gradients.  Also reports the NVFP4 error against the
    BF16 (cuBLAS) product of the same layer, as a sanity bound, not a parity gate."""
    from nvfp4_bit_quantized_gb300 import inputs
    X, W, dY = inputs.heavy_tailed_layer(16384, 4096, 14336, seed=0, device="cuda")
    _layer(nv, oracle_mod, X, W, dY, seed=2)
    wq = nv.quantize_weight(W)
    Y = nv.linear_fprop(X, wq)
    ref = X @ W.t()
    err = ((Y.float() - ref.float()).norm() / ref.float().norm()).item()
    assert err < 0.25, err


@pytest.mark.parametrize("C", [5120, 20480])
def test_quantizer_sweep_largest(nv, oracle_mod, C):
    """The quantizer sweep at 2^28 elements (bf16, 0.1% outlier columns x100), all
    four modes, bit for bit on sampled rows."""
    from nvfp4_bit_quantized_gb300 import inputs
    R = inputs.sweep_rows(28, C)
    x = inputs.sweep_tensor(R, C, seed=3, device="cuda")
    xh = host_input(x)
    rng = np.random.default_rng(C)
    o = oracle_mod
    for block, rnd, rht in ((o.ROW, o.RNE, False), (o.ROW, o.SR, False), (o.TILE16, o.RNE, False),
                            (o.COL, o.SR, True)):
        q = nv.quantize(x, block, rnd, rht=rht, sr_seed=5, sr_offset=1, rht_seed=9, transpose=False)
        _check_operand(o, q, xh, block, rnd, rht, 5, 1, 9, [rng.integers(0, q.rows)])
        del q
        torch.cuda.empty_cache()
