"""The oracle's threaded variants (used only to time it on all host cores) give the
single-threaded results bit for bit: every element's arithmetic is the same, only the
rows are split among threads.  CPU only."""
import numpy as np
import pytest
import torch


def _bits(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("threads", [2, 3, 7, 64])
@pytest.mark.parametrize("mode", ["row_rne", "row_sr", "col_rht_sr", "col_rne", "tile16"])
def test_quantize_mt_equals_single_thread(oracle_mod, mode, threads):
    om = oracle_mod
    kw = dict(row_rne=dict(block=om.ROW), row_sr=dict(block=om.ROW, round_mode=om.SR, sr_seed=5, sr_offset=3),
              col_rht_sr=dict(block=om.COL, round_mode=om.SR, rht=True, sr_seed=5, rht_seed=9),
              col_rne=dict(block=om.COL), tile16=dict(block=om.TILE16))[mode]
    x = _bits((48, 96), 11)                          # 48 operand rows (96 for col): fewer than 64 threads
    x[3, 5] = 0x4F80                                 # an outlier owned by one thread sets the tensor amax
    a = om.quantize(x, **kw)
    b = om.quantize(x, threads=threads, **kw)
    assert np.array_equal(a["codes"], b["codes"]) and np.array_equal(a["scales"], b["scales"])
    assert a["s_dec"] == b["s_dec"] and a["amax"] == b["amax"]
    # a row range: encoded rows only, amax over the whole operand
    lo, hi = (16, 32) if mode == "tile16" else (5, 29)
    c = om.quantize(x, row_begin=lo, row_end=hi, threads=threads, **kw)
    d = om.quantize(x, row_begin=lo, row_end=hi, **kw)
    assert np.array_equal(c["codes"], d["codes"]) and np.array_equal(c["scales"], d["scales"])


def test_quantize_mt_rejects_nonfinite_like_single_thread(oracle_mod):
    x = _bits((32, 64), 2)
    x[31, 63] = 0x7F80                               # +inf in the last thread's rows
    with pytest.raises(FloatingPointError):
        oracle_mod.quantize(x, oracle_mod.ROW, threads=4)


@pytest.mark.parametrize("threads", [2, 5, 16])
def test_gemm_mt_equals_single_thread(oracle_mod, threads):
    rng = np.random.default_rng(3)
    A, B = rng.standard_normal((37, 160)), rng.standard_normal((23, 160))
    assert np.array_equal(oracle_mod.gemm_f64(A, B), oracle_mod.gemm_f64(A, B, threads=threads))
