"""The statistical cost of the SR random-bit layout (elements 4k and 4k+1 draw on one
16-bit value R, the second bit-reversed; likewise 4k+2 and 4k+3): measured against fully
independent 16-bit draws.  CPU only; the oracle's SR rule and bit layout are the ones the
GPU is pinned to bit for bit.  The page's reason for SR is unbiased gradients (page ¶2, ¶4)."""
import numpy as np
import torch

from nvfp4_bit_quantized_gb300 import inputs


def _rev16(v):
    r = np.zeros_like(v)
    for b in range(16):
        r |= ((v >> b) & 1) << (15 - b)
    return r


def test_paired_round_up_decisions_are_nearly_uncorrelated():
    """Exactly, over all 2^16 values of R: the round-up events {R >= T1} and {rev(R) >= T2}
    have |covariance| below 1e-4 for every pair of thresholds on a 257-step grid, against
    variances up to 0.25: the pairing leaves each element's SR unbiased and the pair
    practically independent."""
    R = np.arange(65536, dtype=np.uint32)
    rv = _rev16(R)
    T = np.arange(0, 65537, 257)
    up1 = (R[None, :] >= T[:, None]).astype(np.float64)
    up2 = (rv[None, :] >= T[:, None]).astype(np.float64)
    cov = up1 @ up2.T / 65536 - np.outer(up1.mean(1), up2.mean(1))
    assert np.abs(cov).max() < 1e-4


def test_block_sum_sr_error_variance_paired_vs_independent(oracle_mod):
    """On blocks of heavy-tailed gradients (Student-t(4) as in the heavy-tailed layer),
    scaled so each block's maximum maps to 6 as the encoder does, the variance of the
    16-element block-sum SR error over 256 draws is the same with the paired bits of the
    layout as with independent 16-bit draws (ratio within 3 %), and both are unbiased."""
    om = oracle_mod
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])
    nb, draws = 1500, 256
    g = inputs.student_t((nb, 16), 4, 5, dtype=torch.float32).numpy()
    y = (g * (6.0 / np.abs(g).max(axis=1, keepdims=True))).astype(np.float32)   # block amax -> 6
    idx = np.arange(nb * 16, dtype=np.uint64)
    var = {}
    for layout in ("paired", "independent"):
        sums = np.empty((draws, nb))
        for s in range(draws):
            if layout == "paired":       # the layout: element i draws on word (i >> 2) & 3 of call i >> 4
                r = om.sr_bits(seed=11, stream=0, offset=s, idx=idx)
            else:                        # every element from its own Philox call (word 0, first half)
                r = om.sr_bits(seed=11, stream=0, offset=s, idx=idx * 16)
            q = grid[om.e2m1_encode_sr(y.reshape(-1), r)].reshape(nb, 16)
            sums[s] = (q - y).sum(axis=1)
        # unbiased: the grand mean error is within 4 standard errors of 0
        assert abs(sums.mean()) < 4 * sums.std() / np.sqrt(sums.size)
        var[layout] = sums.var(axis=0).mean()
    ratio = var["paired"] / var["independent"]
    print(f"block-sum SR error variance: paired {var['paired']:.4f}, independent {var['independent']:.4f}, "
          f"ratio {ratio:.4f}")
    assert 0.97 < ratio < 1.03, ratio
