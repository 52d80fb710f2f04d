"""Quantizer parity: the CUDA kernels against the oracle, bit for bit (codes,
canonical and tensor-core-layout scales, the FP32 tensor scale), SR included."""
import numpy as np
import pytest
import torch

from helpers import host_input, mma_layout_from_canonical

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_bit_quantized_gb300 as nv
    return nv


MODES = {
    "row_rne": dict(block=0, round=0, rht=False),
    "row_sr": dict(block=0, round=1, rht=False),
    "col_rne": dict(block=1, round=0, rht=False),
    "col_sr": dict(block=1, round=1, rht=False),
    "col_rht_rne": dict(block=1, round=0, rht=True),
    "col_rht_sr": dict(block=1, round=1, rht=True),
    "tile_rne": dict(block=2, round=0, rht=False),
    "tile_sr": dict(block=2, round=1, rht=False),
}


def _input(shape, dtype, seed, std=1.0, outliers=True):
    from nvfp4_bit_quantized_gb300 import inputs
    x = inputs.normal(shape, std, seed, dtype=torch.float32, device="cpu")
    if outliers:
        inputs.outlier_columns(x, 0.01, 100.0, seed + 7)
    return x.to(dtype)


def check_against_oracle(nv, oracle_mod, x_gpu, mode, sr_seed=0, sr_offset=0, rht_seed=1):
    m = MODES[mode]
    q = nv.quantize(x_gpu, m["block"], m["round"], rht=m["rht"], sr_seed=sr_seed, sr_offset=sr_offset,
                    rht_seed=rht_seed)
    torch.cuda.synchronize()
    xh = host_input(x_gpu)
    ref = oracle_mod.quantize(xh, m["block"], m["round"], rht=m["rht"], sr_seed=sr_seed, sr_offset=sr_offset,
                              rht_seed=rht_seed)
    got_codes = q.codes.cpu().numpy()
    bad = np.argwhere(got_codes != ref["codes"])
    assert bad.size == 0, f"{mode}: {len(bad)} code bytes differ, first {bad[:5].tolist()}"
    assert np.array_equal(q.scales.cpu().numpy(), ref["scales"]), mode
    assert np.float32(q.s_dec[0].item()).tobytes() == np.float32(ref["s_dec"]).tobytes(), mode
    tile = m["block"] == 2
    exp_mma = mma_layout_from_canonical(ref["scales"], q.rows, q.cols, tile2d=tile)
    assert np.array_equal(q.scales_mma.cpu().numpy()[:exp_mma.size], exp_mma), mode
    if tile:
        refT = oracle_mod.quantize(np.ascontiguousarray(xh.T), 2, m["round"], sr_seed=sr_seed, sr_offset=sr_offset)
        if m["round"] == 0:      # RNE: the transposed copy is W^T's own quantization
            assert np.array_equal(q.codes_t.cpu().numpy(), refT["codes"])
        exp_t = mma_layout_from_canonical(ref["scales"].T.copy(), q.cols, q.rows, tile2d=True)
        assert np.array_equal(q.scales_mma_t.cpu().numpy()[:exp_t.size], exp_t)
    return q, ref


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", [(16, 16), (208, 336), (512, 1024)])
def test_quantize_parity(nv, oracle_mod, mode, dtype, shape):
    x = _input(shape, dtype, seed=hash((mode, shape)) % 1000).cuda()
    check_against_oracle(nv, oracle_mod, x, mode, sr_seed=12345, sr_offset=3, rht_seed=77)


@pytest.mark.parametrize("mode", ["row_rne", "row_sr"])
def test_row_mode_ragged_rows_and_pitch(nv, oracle_mod, mode):
    base = _input((37, 400), torch.bfloat16, seed=3).cuda()
    x = base[:, :320]                                   # row pitch 400 > C = 320
    check_against_oracle(nv, oracle_mod, x, mode, sr_seed=9)
    check_against_oracle(nv, oracle_mod, _input((1, 16), torch.bfloat16, 4).cuda(), mode)


@pytest.mark.parametrize("mode", ["col_rht_sr", "tile_rne"])
def test_strided_input(nv, oracle_mod, mode):
    base = _input((96, 512), torch.bfloat16, seed=5).cuda()
    check_against_oracle(nv, oracle_mod, base[:, 64:320], mode, sr_seed=2)


def test_sweep_shape_small(nv, oracle_mod):
    """The quantizer-sweep workload at its smallest size: bf16 [R, 5120], 0.1% outlier columns x100."""
    from nvfp4_bit_quantized_gb300 import inputs
    C = 5120
    R = inputs.sweep_rows(20, C)
    x = inputs.sweep_tensor(R, C, seed=0).cuda()
    for mode in ("row_rne", "row_sr", "tile_rne", "col_rht_sr"):
        check_against_oracle(nv, oracle_mod, x, mode, sr_seed=0, rht_seed=1)


def test_zero_and_signed_zero_inputs(nv, oracle_mod):
    z = torch.zeros((32, 64), dtype=torch.bfloat16, device="cuda")
    z[3, :] = -0.0
    for mode in MODES:
        q, ref = check_against_oracle(nv, oracle_mod, z, mode)
        assert q.s_dec[0].item() == 1.0


def test_empty_input_writes_unit_scale(nv):
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    q = nv.quantize(x, nv.ROW)
    torch.cuda.synchronize()
    assert q.s_dec[0].item() == 1.0


def test_nonfinite_input_sets_device_status(nv):
    for mode in ("row_rne", "col_rht_sr", "tile_rne"):
        m = MODES[mode]
        x = torch.randn((64, 128), device="cuda").to(torch.bfloat16)
        x[5, 7] = float("inf") if mode != "tile_rne" else float("nan")
        nv.reset_status()
        nv.quantize(x, m["block"], m["round"], rht=m["rht"])
        assert nv.status_query() == 7
        nv.reset_status()


def test_sr_seed_and_offset_change_only_codes(nv):
    x = torch.randn((64, 256), device="cuda").to(torch.bfloat16) * 1e-3
    a = nv.quantize(x, nv.ROW, nv.SR, sr_seed=1)
    b = nv.quantize(x, nv.ROW, nv.SR, sr_seed=1)
    c = nv.quantize(x, nv.ROW, nv.SR, sr_seed=1, sr_offset=1)
    torch.cuda.synchronize()
    assert torch.equal(a.codes, b.codes) and not torch.equal(a.codes, c.codes)
    assert torch.equal(a.scales, c.scales)


@pytest.mark.parametrize("mode", ["row_rne", "row_sr"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_row_mode_16_byte_aligned_input(nv, oracle_mod, mode, dtype):
    """Inputs whose blocks start 16 (not 32) bytes apart from a 32-byte boundary take
    the 16-byte load path of the row kernel."""
    base = _input((40, 8 + 16 * 20), dtype, seed=6).cuda()
    off = 8 if dtype == torch.bfloat16 else 4           # 16 bytes
    x = base[:, off:off + 16 * 20]
    assert (x.data_ptr() % 32) == 16
    check_against_oracle(nv, oracle_mod, x, mode, sr_seed=4)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape", [(208, 336), (1024, 512), (64, 4096)])
@pytest.mark.parametrize("rnd,rht", [(0, True), (1, True), (0, False), (1, False)])
def test_dual_quantization_matches_two_single_calls(nv, oracle_mod, dtype, shape, rnd, rht):
    """nvfp4_quantize_dual (one amax read for both operands) == two nvfp4_quantize calls,
    and both operands equal the oracle."""
    x = _input(shape, dtype, seed=sum(shape) + rnd).cuda()
    qr, qc = nv.quantize_dual(x, rnd, rnd, rht=rht, sr_seed=31, sr_offset=2, rht_seed=8)
    ar = nv.quantize(x, nv.ROW, rnd, sr_seed=31, sr_offset=2)
    ac = nv.quantize(x, nv.COL, rnd, rht=rht, sr_seed=31, sr_offset=2, rht_seed=8)
    torch.cuda.synchronize()
    for d, s in ((qr, ar), (qc, ac)):
        assert torch.equal(d.codes, s.codes) and torch.equal(d.scales, s.scales)
        assert torch.equal(d.scales_mma, s.scales_mma) and torch.equal(d.s_dec[:1], s.s_dec[:1])
    xh = host_input(x)
    r = oracle_mod.quantize(xh, oracle_mod.ROW, rnd, sr_seed=31, sr_offset=2)
    c = oracle_mod.quantize(xh, oracle_mod.COL, rnd, rht=rht, sr_seed=31, sr_offset=2, rht_seed=8)
    assert np.array_equal(qr.codes.cpu().numpy(), r["codes"]) and np.array_equal(qc.codes.cpu().numpy(), c["codes"])


@pytest.mark.parametrize("rnd_row,rnd_col", [(1, 0), (0, 1), (1, 1), (0, 0)])
def test_dual_quantization_mixed_rounding_and_seeds(nv, oracle_mod, rnd_row, rnd_col):
    """Row and column operands with different SR seeds and offsets, with different rounding
    modes (two encode kernels) and with one mode for both (the fused encode)."""
    x = _input((192, 320), torch.bfloat16, seed=77).cuda()
    qr, qc = nv.quantize_dual(x, rnd_row, rnd_col, rht=True, sr_seed=11, sr_offset=5, rht_seed=6,
                              col_sr_seed=23, col_sr_offset=9)
    torch.cuda.synchronize()
    xh = host_input(x)
    r = oracle_mod.quantize(xh, oracle_mod.ROW, rnd_row, sr_seed=11, sr_offset=5)
    c = oracle_mod.quantize(xh, oracle_mod.COL, rnd_col, rht=True, sr_seed=23, sr_offset=9, rht_seed=6)
    assert np.array_equal(qr.codes.cpu().numpy(), r["codes"]) and np.array_equal(qr.scales.cpu().numpy(), r["scales"])
    assert np.array_equal(qc.codes.cpu().numpy(), c["codes"]) and np.array_equal(qc.scales.cpu().numpy(), c["scales"])
