"""The synthetic workload recipe (seeded inputs shared by the tests and the bench): shapes,
determinism, the outlier structure and the distributions, checked on the CPU."""
import math

import numpy as np
import torch

from nvfp4_bit_quantized_gb300 import inputs


def test_seeded_and_deterministic():
    a = inputs.normal((64, 32), 0.02, 5)
    b = inputs.normal((64, 32), 0.02, 5)
    c = inputs.normal((64, 32), 0.02, 6)
    assert a.dtype == torch.bfloat16 and torch.equal(a, b) and not torch.equal(a, c)
    X, W, dY = inputs.linear_layer(32, 48, 64, seed=0)
    assert X.shape == (32, 48) and W.shape == (64, 48) and dY.shape == (32, 64)
    assert torch.equal(X, inputs.normal((32, 48), 1.0, 0)) and torch.equal(W, inputs.normal((64, 48), 0.02, 1))


def test_normal_moments():
    x = inputs.normal((512, 512), 1e-3, 9, dtype=torch.float32).double()
    assert abs(x.mean().item()) < 1e-5 and abs(x.std().item() / 1e-3 - 1) < 0.01


def test_sweep_shapes_and_outlier_columns():
    for p in (20, 24, 28):
        for C in (5120, 20480):
            R = inputs.sweep_rows(p, C)
            assert R % 16 == 0 and R >= 16 and abs(R * C - 2 ** p) <= 8 * C + 1
    x = inputs.sweep_tensor(256, 5120, seed=3).float()
    col_rms = x.pow(2).mean(dim=0).sqrt()
    big = (col_rms > 20).nonzero().flatten()
    assert len(big) == round(0.001 * 5120)                     # 5 columns x100
    assert torch.all((col_rms[big] > 60) & (col_rms[big] < 140))


def test_heavy_tailed_layer_structure():
    X, W, dY = inputs.heavy_tailed_layer(4096, 4096, 256, seed=0)
    assert X.shape == (4096, 4096) and W.shape == (256, 4096) and dY.shape == (4096, 256)
    xf = X.float()
    med = xf.abs().median(dim=0).values
    big = (med > 10 * med.median()).nonzero().flatten()
    assert len(big) == round(0.01 * 4096)                      # 41 channels x50
    # Student-t(3) on the other channels: heavier tails than a normal of the same spread
    rest = xf[:, [c for c in range(4096) if c not in set(big.tolist())][:256]].flatten().double()
    kurt = ((rest - rest.mean()) ** 4).mean() / rest.var() ** 2
    assert kurt > 6                                            # a normal's kurtosis is 3
    g = dY.float().flatten().double()
    assert abs(g.std().item() / 1e-3 - math.sqrt(2)) < 0.2     # t(4) has variance 4 / (4 - 2) = 2


def test_token_outlier_layer_structure():
    """Outliers along the tokens: the same 1% of rows of X and dY are x50, no channel is."""
    X, W, dY = inputs.heavy_tailed_token_outliers(2048, 512, 384, seed=0)
    assert X.shape == (2048, 512) and W.shape == (384, 512) and dY.shape == (2048, 384)
    rx = X.float().abs().median(dim=1).values
    rg = dY.float().abs().median(dim=1).values
    bx = set((rx > 10 * rx.median()).nonzero().flatten().tolist())
    bg = set((rg > 10 * rg.median()).nonzero().flatten().tolist())
    assert len(bx) == round(0.01 * 2048) and bx == bg              # 20 tokens, the same in X and dY
    cx = X.float().abs().median(dim=0).values
    assert (cx > 10 * cx.median()).sum() == 0                      # no outlier channels
