"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- the format definitions, a library routine, brute force, exact
arithmetic, or an invariant the news page states.  CPU only.

Page: "NVIDIA NVFP4 paper: 4-bit pretrain hits FP8 parity (12B, 10T tokens)"
(zubnet.ai), cited as [page ¶n].
"""
import ctypes
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
FACTS = json.load(open(os.path.join(HERE, "golden", "page_facts.json")))


def f32(x):
    return np.float32(x)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- E2M1 grid ----

def test_e2m1_decode_matches_bitfield_definition(oracle_mod):
    # E2M1: sign | 2 exponent bits (bias 1) | 1 mantissa bit; exponent 0 is subnormal.
    for code in range(16):
        s, e, m = code >> 3, (code >> 1) & 3, code & 1
        mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        assert oracle_mod.e2m1_value(code) == (-mag if s else mag)
    grid = sorted({abs(oracle_mod.e2m1_value(c)) for c in range(16)})
    assert grid == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert FACTS["element_format"]["value"] == "E2M1"


# ---------------------------------------------------------------- E4M3 --------

def test_e4m3_decode_matches_torch(oracle_mod):
    codes = torch.arange(256, dtype=torch.int16).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle_mod.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v)
        else:
            assert v == ref[c], c


def _brute_e4m3(v: float) -> int:
    """Nearest finite non-negative E4M3 code by exhaustive search; ties -> even code; saturating."""
    best, bd = 0, None
    for c in range(0x7F):              # 0x00..0x7E: all finite non-negative codes
        d = abs(Fraction(float(v)) - Fraction(oracle_val_e4m3(c)))
        if bd is None or d < bd or (d == bd and c % 2 == 0):
            best, bd = c, d
    return best


_E4M3 = None


def oracle_val_e4m3(c):
    global _E4M3
    if _E4M3 is None:
        t = torch.arange(256, dtype=torch.int16).to(torch.uint8).view(torch.float8_e4m3fn)
        _E4M3 = t.to(torch.float64).tolist()
    return _E4M3[c]


def test_e4m3_encode_brute_force(oracle_mod):
    pts = [oracle_val_e4m3(c) for c in range(0x7F)]
    vals = set()
    for a, b in zip(pts[:-1], pts[1:]):
        mid = (a + b) / 2
        vals.update([a, b, mid, np.nextafter(f32(mid), f32(0)), np.nextafter(f32(mid), f32(1e9))])
    vals.update([2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11, 448, 449, 464, 465, 1e6, 0.0])
    rng = np.random.default_rng(0)
    vals.update(rng.uniform(0, 460, 300).tolist())
    vals.update((2.0 ** rng.uniform(-12, -5, 200)).tolist())
    v = np.array(sorted(vals), dtype=np.float32)
    got = oracle_mod.e4m3_encode(v)
    for x, g in zip(v, got):
        assert g == _brute_e4m3(float(x)), (float(x), g)


def test_e4m3_encode_matches_torch_cast_in_range(oracle_mod):
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.uniform(0, 448, 20000), 2.0 ** rng.uniform(-12, 8.8, 20000)]).astype(np.float32)
    v = v[v <= 448]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle_mod.e4m3_encode(v), ref)


# ---------------------------------------------------------------- E2M1 encode ---

def _brute_e2m1_rne(y: float) -> int:
    best, bd = 0, None
    for c in range(8):
        d = abs(Fraction(abs(float(y))) - Fraction(abs(float(np.float64([0, .5, 1, 1.5, 2, 3, 4, 6][c])))))
        if bd is None or d < bd or (d == bd and c % 2 == 0):
            best, bd = c, d
    return best | (8 if math.copysign(1.0, y) < 0 else 0)


def test_e2m1_rne_brute_force(oracle_mod):
    grid = [0, .5, 1, 1.5, 2, 3, 4, 6]
    vals = set([-0.0, 0.0, 7.0, -7.0, 1e30, 5.999, 6.0, 6.0001])
    for a, b in zip(grid[:-1], grid[1:]):
        m = (a + b) / 2
        for x in (a, b, m, float(np.nextafter(f32(m), f32(0))), float(np.nextafter(f32(m), f32(9)))):
            vals.update([x, -x])
    rng = np.random.default_rng(2)
    vals.update(rng.uniform(-7, 7, 3000).tolist())
    y = np.array(sorted(vals), dtype=np.float32)
    got = oracle_mod.e2m1_encode_rne(y)
    for x, g in zip(y, got):
        assert g == _brute_e2m1_rne(float(x)), (float(x), g)


# ---------------------------------------------------------------- SR --------------

def test_sr_exact_expectation_by_enumeration(oracle_mod):
    """E[value] over all 2^16 random values equals lo + (hi-lo) * floor(p * 2^16) / 2^16:
    adding a uniform 16-bit fraction of the spacing and truncating rounds up for
    exactly floor(p * 2^16) of the 2^16 values."""
    grid = [0, .5, 1, 1.5, 2, 3, 4, 6]
    r = np.arange(65536, dtype=np.uint32)
    for a in [0.0, 0.1, 0.25, 0.3, 0.5, 0.77, 1.0, 1.2345, 1.99, 2.5, 3.001, 4.0, 4.2, 5.9, 6.0, 7.5]:
        codes = oracle_mod.e2m1_encode_sr(np.full(65536, a, np.float32), r)
        vals = np.array([grid[c & 7] for c in codes])
        a32 = float(f32(a))
        if a32 >= 6:
            assert np.all(vals == 6)
            continue
        lo = max(g for g in grid if g <= a32)
        hi = min(g for g in grid if g > a32)
        p = Fraction(a32) - Fraction(lo)
        p /= Fraction(hi) - Fraction(lo)
        n_up = math.floor(p * 65536)
        expect = Fraction(lo) + (Fraction(hi) - Fraction(lo)) * Fraction(n_up, 65536)
        assert Fraction(int(np.sum(vals * 2)), 2 * 65536) == expect, a
        assert set(np.unique(vals)).issubset({lo, hi})


def test_sr_unbiased_over_philox_draws(oracle_mod):
    """Mean of 10^4 SR draws (distinct counters) is within 3 sigma of the input [page ¶4]."""
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    n = 10000
    bits = oracle_mod.sr_bits(seed=1234, stream=0, offset=0, idx=np.arange(n, dtype=np.uint64))
    for a in [0.3, 1.1, 2.7, 4.9]:
        vals = grid[oracle_mod.e2m1_encode_sr(np.full(n, a, np.float32), bits) & 7]
        lo, hi = grid[grid <= a].max(), grid[grid > a].min()
        p = (a - lo) / (hi - lo)
        sigma = (hi - lo) * math.sqrt(p * (1 - p) / n)
        assert abs(vals.mean() - a) < 3 * sigma + 1e-12, a
        # negative control: round-to-nearest is visibly biased at these points
        rne = grid[oracle_mod.e2m1_encode_rne(np.full(1, a, np.float32)) & 7][0]
        assert abs(rne - a) > 3 * sigma


def test_sr_keeps_grid_points(oracle_mod):
    r = np.arange(0, 65536, 97, dtype=np.uint32)
    for g in [0, .5, 1, 1.5, 2, 3, 4, 6]:
        for s in (1, -1):
            c = oracle_mod.e2m1_encode_sr(np.full(r.size, s * g, np.float32), r)
            assert np.all(np.abs(np.array([oracle_mod.e2m1_value(int(k)) for k in c])) == g)


# ---------------------------------------------------------------- Philox ----------

def _curand():
    for name in ("libcurand.so.10", "/usr/local/cuda/lib64/libcurand.so.10"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    return None


@pytest.mark.parametrize("seed", [0, 7, 0x9ABCDEF012345678])
def test_philox_matches_curand_host_generator(oracle_mod, seed):
    """cuRAND's host PHILOX4_32_10 generator (a library routine, run only) emits, for
    seed s, block j of four words = Philox4x32-10(key=(lo32 s, hi32 s),
    ctr=(j >> 16, 0, j & 0xFFFF, 0)); compare 70000 blocks with the oracle."""
    lib = _curand()
    if lib is None:
        pytest.skip("libcurand not available")
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0   # PHILOX4_32_10
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        nblk = 70000
        buf = np.zeros(4 * nblk, dtype=np.uint32)
        assert lib.curandGenerate(gen, buf.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(buf.size)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    ref = buf.reshape(nblk, 4)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for j in list(range(0, 300)) + list(range(65530, 65542)) + list(range(69990, 70000)):
        got = oracle_mod.philox4x32_10([j >> 16, 0, j & 0xFFFF, 0], key)
        assert np.array_equal(got, ref[j]), j


def test_sr_bits_uniform_chi_square(oracle_mod):
    n = 1 << 18
    r = oracle_mod.sr_bits(seed=99, stream=1, offset=3, idx=np.arange(n, dtype=np.uint64))
    assert r.max() < 65536
    hist = np.bincount(r >> 10, minlength=64)           # 64 bins
    exp = n / 64
    chi2 = float(((hist - exp) ** 2 / exp).sum())
    assert chi2 < 120.0                                  # 63 dof: p ~ 1e-5 cut
    # streams and offsets give different bits
    r2 = oracle_mod.sr_bits(seed=99, stream=0, offset=3, idx=np.arange(64, dtype=np.uint64))
    r3 = oracle_mod.sr_bits(seed=99, stream=1, offset=4, idx=np.arange(64, dtype=np.uint64))
    assert not np.array_equal(r[:64], r2) and not np.array_equal(r[:64], r3)


def test_sr_bits_layout_in_philox_words(oracle_mod):
    """One Philox call per 16 elements; elements 4k..4k+3 split word k into
    A = bytes (2, 0), A reversed, B = bytes (3, 1), B reversed."""
    seed = 0x0123456789ABCDEF
    idx = np.arange(96, dtype=np.uint64)
    got = oracle_mod.sr_bits(seed, 1, 5, idx)

    def rev16(v):
        return int(format(v, "016b")[::-1], 2)

    for i in range(96):
        w = oracle_mod.philox4x32_10([i >> 4, 0, 1, 5], [seed & 0xFFFFFFFF, seed >> 32])
        word = int(w[(i >> 2) & 3])
        a = (((word >> 16) & 0xFF) << 8) | (word & 0xFF)
        b = (((word >> 24) & 0xFF) << 8) | ((word >> 8) & 0xFF)
        assert got[i] == [a, rev16(a), b, rev16(b)][i & 3], i


def test_sr_decisions_of_paired_elements_are_unbiased(oracle_mod):
    """Elements 4k and 4k+1 draw on the same 16 bits (one reversed): each is still
    exactly uniform, so each element's SR stays unbiased; and the pair is not
    degenerate (both round-up events occur together about p^2 of the time)."""
    n = 1 << 16
    bits = oracle_mod.sr_bits(seed=5, stream=0, offset=0, idx=np.arange(4 * n, dtype=np.uint64)).reshape(n, 4)
    for c in range(4):
        hist = np.bincount(bits[:, c] >> 12, minlength=16)
        assert float(((hist - n / 16) ** 2 / (n / 16)).sum()) < 45.0        # 15 dof
    y = np.full(n, 1.3, np.float32)                                      # p = 0.6 on [1, 1.5)
    up0 = oracle_mod.e2m1_encode_sr(y, bits[:, 0]) == 3
    up1 = oracle_mod.e2m1_encode_sr(y, bits[:, 1]) == 3
    for u in (up0, up1):
        assert abs(u.mean() - 0.6) < 4 * math.sqrt(0.24 / n)
    assert abs((up0 & up1).mean() - 0.36) < 0.02


# ---------------------------------------------------------------- RHT --------------

def test_hadamard_stage_product_is_sylvester(oracle_mod):
    import scipy.linalg
    H = oracle_mod.hadamard_stage_product()
    assert np.array_equal(H, scipy.linalg.hadamard(16))
    assert np.array_equal(H @ H.T, 16 * np.eye(16, dtype=np.int64))
    assert FACTS["hadamard_size"]["value"] == 16


def test_rht16_matches_dense_product_and_inverts(oracle_mod):
    import scipy.linalg
    H = scipy.linalg.hadamard(16).astype(np.float64)
    rng = np.random.default_rng(3)
    for trial in range(200):
        v = (rng.standard_normal(16) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
        mask = int(rng.integers(0, 1 << 16))
        s = np.array([-1.0 if (mask >> j) & 1 else 1.0 for j in range(16)])
        y = oracle_mod.rht16(v, mask).astype(np.float64)
        dense = H @ (s * v.astype(np.float64)) / 4.0
        bound = 4 * 2.0 ** -24 * np.abs(v.astype(np.float64)).sum()       # 4 roundings per entry
        assert np.all(np.abs(y - dense) <= bound)
        # R^T (R v) = v: R^T = diag(s) H / 4
        back = s * (H @ y) / 4.0
        assert np.allclose(back, v, rtol=0, atol=8 * 2.0 ** -24 * np.abs(v).sum())
    # all-positive signs reduce to the plain (scaled) Walsh-Hadamard transform
    v = rng.standard_normal(16).astype(np.float32)
    y = oracle_mod.rht16(v, 0).astype(np.float64)
    assert np.allclose(y, H @ v.astype(np.float64) / 4, atol=1e-6)


def test_rht16_zero_signs_and_exact_cases(oracle_mod):
    # a single impulse maps to a signed row of H / 4 exactly
    import scipy.linalg
    H = scipy.linalg.hadamard(16)
    for j in range(16):
        v = np.zeros(16, np.float32)
        v[j] = 4.0
        y = oracle_mod.rht16(v, 1 << j)
        assert np.array_equal(y, -H[:, j].astype(np.float32))


def test_rht_sign_mask_is_philox_word0(oracle_mod):
    for seed in (1, 2, 12345):
        w = oracle_mod.philox4x32_10([0, 0, 0, 0], [seed & 0xFFFFFFFF, seed >> 32])
        assert oracle_mod.rht_sign_mask(seed) == int(w[0]) & 0xFFFF


# ---------------------------------------------------------------- quantize ---------

def _rand_bf16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


def test_tensor_scale_closed_form_and_power_of_two_invariance(oracle_mod):
    x = torch.randn(64, 48, generator=torch.Generator().manual_seed(5)).numpy().astype(np.float32)
    q = oracle_mod.quantize(x, oracle_mod.ROW)
    amax = float(np.abs(x).max())
    assert q["amax"] == amax
    s_enc = f32(f32(2688.0) / f32(amax))
    assert q["s_dec"] == float(f32(1.0) / s_enc)
    for k in (-7, -1, 3, 9):
        q2 = oracle_mod.quantize((x * f32(2.0 ** k)).astype(np.float32), oracle_mod.ROW)
        assert np.array_equal(q2["codes"], q["codes"]) and np.array_equal(q2["scales"], q["scales"])
        assert q2["s_dec"] == q["s_dec"] * 2.0 ** k
    z = oracle_mod.quantize(np.zeros((16, 32), np.float32), oracle_mod.ROW)
    assert z["s_dec"] == 1.0 and not z["codes"].any() and not z["scales"].any()


def test_block_scale_is_nearest_e4m3(oracle_mod):
    x = _rand_bf16((32, 256), 6)
    xb = bf16_bits(x)
    q = oracle_mod.quantize(xb, oracle_mod.ROW)
    xf = x.float().numpy()
    s_enc = f32(f32(2688.0) / f32(np.abs(xf).max()))
    for r in range(0, 32, 3):
        for b in range(16):
            amax_b = f32(np.abs(xf[r, 16 * b:16 * b + 16]).max())
            t = f32(f32(amax_b / f32(6.0)) * s_enc)
            assert q["scales"][r, b] == _brute_e4m3(float(t))


def test_brute_force_tile_encode(oracle_mod):
    """Enumerate all 16 codes for every element of 16x16 tiles: the oracle's code is
    the nearest to y = x * e_b (ties to even), with the block scale's multiplier."""
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])
    x = _rand_bf16((16, 64), 7)
    xf = x.float().numpy()
    for mode in (oracle_mod.ROW, oracle_mod.TILE16):
        q = oracle_mod.quantize(bf16_bits(x), mode)
        s_enc = f32(f32(2688.0) / f32(np.abs(xf).max()))
        for i in range(16):
            for j in range(64):
                sb = q["scales"][i, j // 16] if mode == oracle_mod.ROW else q["scales"][0, j // 16]
                e_b = f32(s_enc / f32(oracle_val_e4m3(int(sb))))
                y = f32(f32(xf[i, j]) * e_b)
                code = (q["codes"][i, j // 2] >> (4 * (j & 1))) & 15
                d = np.abs(grid - min(abs(float(y)), 6.0) * np.sign(float(y) or 1.0))
                best = [c for c in range(16) if d[c] == d.min()]
                if len(best) > 1:       # tie or zero: choose the even magnitude with the input's sign
                    best = [c for c in best if (c & 1) == 0 and ((c >> 3) == (1 if math.copysign(1, y) < 0 else 0))]
                assert code == best[0], (mode, i, j, float(y), code, best)


@pytest.mark.parametrize("mode", ["row", "col", "col_rht", "tile"])
def test_amax_element_is_at_scale_precision(oracle_mod, mode):
    """[page ¶2] one value in sixteen per block (6.25 %) keeps roughly FP8 precision: with
    RNE, the block's largest element encodes to +-6 whenever the block scale is normal."""
    frac = FACTS["min_fraction_at_scale_precision"]["value"]
    assert frac == 1 / FACTS["block_elems"]["value"]
    x = _rand_bf16((64, 128), 8)
    xf = x.float().numpy().astype(np.float64)
    kw = dict(row=dict(block=oracle_mod.ROW), col=dict(block=oracle_mod.COL),
              col_rht=dict(block=oracle_mod.COL, rht=True, rht_seed=1),
              tile=dict(block=oracle_mod.TILE16))[mode]
    q = oracle_mod.quantize(bf16_bits(x), **kw)
    codes = np.stack([q["codes"] & 15, q["codes"] >> 4], -1).reshape(q["rows"], q["cols"])
    if mode == "col_rht":
        T = np.stack([oracle_mod.rht16(c, oracle_mod.rht_sign_mask(1)) for c in
                      x.float().numpy().T.reshape(-1, 16)]).reshape(q["rows"], q["cols"])
    else:
        T = xf.T if mode == "col" else xf
    bh = 16 if mode == "tile" else 1
    checked = 0
    for i0 in range(0, q["rows"], bh):
        for j0 in range(0, q["cols"], 16):
            blk = np.abs(T[i0:i0 + bh, j0:j0 + 16])
            sb = q["scales"][i0 // 16, j0 // 16] if mode == "tile" else q["scales"][i0, j0 // 16]
            if oracle_val_e4m3(int(sb)) < 2.0 ** -6:
                continue
            ii, jj = np.unravel_index(np.argmax(blk), blk.shape)
            assert codes[i0 + ii, j0 + jj] & 7 == 7
            checked += 1
    assert checked > 0


def test_2d_weights_same_representation_both_ways(oracle_mod):
    """[page ¶2] 2D weight scaling: W and W^T dequantize identically, bit for bit;
    negative control: 1x16 row scaling does not."""
    W = _rand_bf16((64, 96), 9, std=0.02)
    qa = oracle_mod.quantize(bf16_bits(W), oracle_mod.TILE16)
    qb = oracle_mod.quantize(bf16_bits(W.t().contiguous()), oracle_mod.TILE16)
    assert np.array_equal(oracle_mod.dequant(qa).T, oracle_mod.dequant(qb))
    ra = oracle_mod.quantize(bf16_bits(W), oracle_mod.ROW)
    rb = oracle_mod.quantize(bf16_bits(W.t().contiguous()), oracle_mod.ROW)
    assert not np.array_equal(oracle_mod.dequant(ra).T, oracle_mod.dequant(rb))


def test_col_mode_is_row_mode_of_transpose(oracle_mod):
    """Without RHT and SR, 1x16 column quantization of X equals row quantization of X^T."""
    x = _rand_bf16((48, 80), 10)
    qc = oracle_mod.quantize(bf16_bits(x), oracle_mod.COL)
    qr = oracle_mod.quantize(bf16_bits(x.t().contiguous()), oracle_mod.ROW)
    assert np.array_equal(qc["codes"], qr["codes"]) and np.array_equal(qc["scales"], qr["scales"])
    assert qc["s_dec"] == qr["s_dec"]


def test_rht_wgrad_identity_and_sign_sharing(oracle_mod):
    """(R dY)^T (R X) = dY^T X: with the RHT on both Wgrad operands (same signs) the
    product of the transformed operands equals the plain product up to rounding."""
    M, N, K = 64, 32, 48
    dY = np.random.default_rng(11).standard_normal((M, N)).astype(np.float32)
    X = np.random.default_rng(12).standard_normal((M, K)).astype(np.float32)
    mask = oracle_mod.rht_sign_mask(1)
    RdY = np.stack([oracle_mod.rht16(c, mask) for c in dY.T.reshape(-1, 16)]).reshape(N, M)
    RX = np.stack([oracle_mod.rht16(c, mask) for c in X.T.reshape(-1, 16)]).reshape(K, M)
    exact = dY.T.astype(np.float64) @ X.astype(np.float64)
    got = RdY.astype(np.float64) @ RX.astype(np.float64).T
    assert np.abs(got - exact).max() < 1e-4
    other = oracle_mod.rht_sign_mask(2)
    RX2 = np.stack([oracle_mod.rht16(c, other) for c in X.T.reshape(-1, 16)]).reshape(K, M)
    assert np.abs(RdY.astype(np.float64) @ RX2.astype(np.float64).T - exact).max() > 1.0


def test_sr_mode_uses_only_neighbours(oracle_mod):
    x = _rand_bf16((32, 64), 13, std=1e-3)
    q1 = oracle_mod.quantize(bf16_bits(x), oracle_mod.ROW, oracle_mod.SR, sr_seed=5)
    q2 = oracle_mod.quantize(bf16_bits(x), oracle_mod.ROW, oracle_mod.SR, sr_seed=5)
    q3 = oracle_mod.quantize(bf16_bits(x), oracle_mod.ROW, oracle_mod.SR, sr_seed=6)
    assert np.array_equal(q1["codes"], q2["codes"])          # reproducible for a seed
    assert not np.array_equal(q1["codes"], q3["codes"])
    assert np.array_equal(q1["scales"], q3["scales"])         # scales do not depend on SR


def test_nonfinite_input_is_rejected(oracle_mod):
    x = np.ones((16, 16), np.float32)
    x[3, 5] = np.inf
    with pytest.raises(FloatingPointError):
        oracle_mod.quantize(x, oracle_mod.ROW)
    x[3, 5] = np.nan
    with pytest.raises(FloatingPointError):
        oracle_mod.quantize(x, oracle_mod.COL)


def test_row_range_matches_full(oracle_mod):
    x = _rand_bf16((80, 64), 14)
    full = oracle_mod.quantize(bf16_bits(x), oracle_mod.COL, oracle_mod.SR, rht=True, sr_seed=3, rht_seed=4)
    part = oracle_mod.quantize(bf16_bits(x), oracle_mod.COL, oracle_mod.SR, rht=True, sr_seed=3, rht_seed=4,
                               row_begin=16, row_end=40)
    assert np.array_equal(full["codes"][16:40], part["codes"][16:40])
    assert np.array_equal(full["scales"][16:40], part["scales"][16:40])


def test_memory_footprint_about_half_of_fp8():
    """[page ¶1] operand memory about halved vs FP8: 4 bits + one 8-bit scale per 16."""
    bits = 4 + 8 / FACTS["block_elems"]["value"]
    assert abs(bits / 8 - FACTS["operand_memory_vs_fp8"]["value"]) <= 0.0625


# ---------------------------------------------------------------- GEMM ---------------

@pytest.mark.parametrize("M,N,K", [(16, 16, 16), (32, 32, 64)])
def test_gemm_f64_against_exact_integer_arithmetic(oracle_mod, M, N, K):
    """2*val(E2M1) and 2^9*val(E4M3) are integers, so the dequantized dot products are
    exact rationals; the fp64 oracle must agree to within K fp64 roundings."""
    A = _rand_bf16((M, K), 15)
    B = _rand_bf16((N, K), 16, std=0.02)
    qa = oracle_mod.quantize(bf16_bits(A), oracle_mod.ROW)
    qb = oracle_mod.quantize(bf16_bits(B), oracle_mod.TILE16)
    C = oracle_mod.gemm_f64(oracle_mod.dequant(qa), oracle_mod.dequant(qb))

    def ints(q, tile):
        codes = np.stack([q["codes"] & 15, q["codes"] >> 4], -1).reshape(q["rows"], q["cols"])
        e2 = np.array([int(2 * v) for v in [0, .5, 1, 1.5, 2, 3, 4, 6]])
        val2 = np.where(codes & 8, -1, 1) * e2[codes & 7]
        sc = q["scales"] if not tile else np.repeat(q["scales"], 16, axis=0)
        s9 = np.vectorize(lambda c: int(round(oracle_val_e4m3(int(c)) * 512)))(sc)
        return val2.astype(object), np.repeat(s9, 16, axis=1).astype(object)

    va, sa = ints(qa, False)
    vb, sb = ints(qb, True)
    sd = Fraction(qa["s_dec"]) * Fraction(qb["s_dec"]) / (4 * 512 * 512)
    for m in range(M):
        for n in range(N):
            terms = [va[m, k] * sa[m, k] * vb[n, k] * sb[n, k] for k in range(K)]
            exact = sum(terms) * sd
            mag = sum(abs(t) for t in terms) * sd
            assert abs(Fraction(C[m, n]) - exact) <= mag * Fraction(K + 2, 2 ** 52), (m, n)


def test_bf16_rounding_helper_matches_torch(oracle_mod):
    """The oracle's fp32 -> bf16 rounding (used by the MLP activation) equals torch's cast."""
    rng = np.random.default_rng(21)
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.uniform(-5, 5, 100000),
                        np.array([0.0, -0.0, 1.0, 3.0e38])]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle_mod._f32_to_bf16(x), ref)


# ---------------------------------------------------------------- squared ReLU (MLP block) --
# The reading (the page names no activation): relu(h) = h if h > 0 else +0 (so -0, negative
# values and NaN give +0); a = relu(h)^2 and dh = da * (2 relu(h)) are each one fp32 operation
# rounded to nearest, then rounded to nearest-even bf16.  The pins below take another route to
# the same numbers: the product of two bf16 values has at most 16 significant bits and an
# exponent far inside fp64's range, so it is exact in fp64; one conversion to fp32 (numpy's
# IEEE cast, which overflows to inf and underflows gradually) is then the single fp32 rounding,
# and torch's fp32 -> bf16 cast is the final rounding (not the oracle's bit arithmetic).

ALL_BF16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def _bf16_as_f64(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def _f32_to_bf16_torch(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def _same_or_both_nan(got: np.ndarray, ref: np.ndarray) -> bool:
    g, r = _bf16_as_f64(got), _bf16_as_f64(ref)
    nan = np.isnan(r)
    return bool(np.array_equal(np.isnan(g), nan) and np.array_equal(got[~nan], ref[~nan]))


def test_sqrelu_forward_all_bf16_patterns(oracle_mod):
    """a = relu(h)^2 for every one of the 65536 bf16 inputs (both zeros, subnormals, the
    fp32 overflow of h^2 above ~1.8e19, inf, NaN): exact square -> one fp32 rounding -> bf16."""
    h = _bf16_as_f64(ALL_BF16)
    with np.errstate(over="ignore", invalid="ignore"):
        pos = h > 0                                  # False for -0, negatives and NaN
        sq = np.where(pos, h * h, 0.0)               # exact in fp64 (or inf for h = inf)
        ref = _f32_to_bf16_torch(sq.astype(np.float32))
        got = oracle_mod.sqrelu_forward(ALL_BF16)
    assert _same_or_both_nan(got, ref)
    # the reading's special cases, spelled out
    assert got[0x0000] == 0 and got[0x8000] == 0                 # relu(+-0)^2 = +0
    assert got[0x7FC0] == 0 and got[0xFFC0] == 0                 # NaN -> +0
    assert got[0x3F80] == 0x3F80 and got[0xBF80] == 0            # 1 -> 1, -1 -> +0
    assert got[0x4040] == 0x4110                                  # 3 -> 9
    assert got[0x7F80] == 0x7F80 and got[0x5F80] == 0x7F80       # inf -> inf; 2^64 squared overflows fp32
    assert got[0x0001] == 0                                       # smallest subnormal: 2^-266 underflows


def _dense_pairs():
    """Every bf16 h against special and random da values, and every bf16 da against
    special and random h values."""
    rng = np.random.default_rng(31)
    special = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x0080, 0x3F80, 0xBF80, 0x4000, 0x3A83,
                        0xBA83, 0x7F7F, 0xFF7F, 0x5F80, 0x5F7F, 0x1F80, 0x2000, 0x7F80, 0xFF80, 0x7FC0,
                        0x0C00, 0x8C00, 0x3C00, 0x4300], dtype=np.uint16)
    rand = rng.integers(0, 65536, 40).astype(np.uint16)
    partners = np.concatenate([special, rand])
    h = np.concatenate([np.repeat(ALL_BF16, partners.size), np.tile(partners, 65536)])
    da = np.concatenate([np.tile(partners, 65536), np.repeat(ALL_BF16, partners.size)])
    return h, da


def test_sqrelu_backward_dense_sweep(oracle_mod):
    """dh = da * 2 relu(h) over ~8.4 M (h, da) pairs: 2h exact then one fp32 rounding (inf
    above the fp32 range), the exact product da * t then one fp32 rounding, then bf16."""
    h_bits, da_bits = _dense_pairs()
    h, da = _bf16_as_f64(h_bits), _bf16_as_f64(da_bits)
    with np.errstate(over="ignore", invalid="ignore"):
        t = np.where(h > 0, 2.0 * h, 0.0).astype(np.float32).astype(np.float64)
        p = da * t                                   # exact for finite t; inf * 0 -> NaN
        ref = _f32_to_bf16_torch(p.astype(np.float32))
        got = oracle_mod.sqrelu_backward(h_bits, da_bits)
    assert _same_or_both_nan(got, ref)
    # spelled-out cases: the gradient through relu is 0 for h <= 0 and keeps da's sign
    one, mone, three = 0x3F80, 0xBF80, 0x4040
    assert oracle_mod.sqrelu_backward(np.array([three], np.uint16), np.array([one], np.uint16))[0] == 0x40C0  # 6
    assert oracle_mod.sqrelu_backward(np.array([mone], np.uint16), np.array([one], np.uint16))[0] == 0x0000
    assert oracle_mod.sqrelu_backward(np.array([mone], np.uint16), np.array([mone], np.uint16))[0] == 0x8000
    with np.errstate(over="ignore"):
        assert oracle_mod.sqrelu_backward(np.array([0x7F7F], np.uint16), np.array([one], np.uint16))[0] == 0x7F80


# ---------------------------------------------------------------- MXFP4 (comparison format) --

def _brute_e2m1_times(y: Fraction) -> Fraction:
    """Nearest E2M1 magnitude to |y| (ties to the even code, > 6 saturates), with y's sign."""
    grid = [Fraction(v) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    a = abs(y)
    if a > 6:
        best = 7
    else:
        best = min(range(8), key=lambda k: (abs(a - grid[k]), k % 2))
    return grid[best] if y >= 0 else -grid[best]


def test_mx_scale_puts_the_block_maximum_in_4_to_8(oracle_mod):
    """The shared exponent maps the block's largest magnitude into [4, 8) (the top E2M1
    binade), the defining property of the MX scale; an all-zero block stores code 0."""
    rng = np.random.default_rng(11)
    vals = list((2.0 ** rng.uniform(-120, 120, 4000)).astype(np.float32))
    vals += [np.float32(2.0 ** k) for k in range(-120, 121)]
    vals += [np.nextafter(np.float32(2.0 ** k), np.float32(0)) for k in range(-120, 121)]
    for a in vals:
        c = oracle_mod.mx_scale_code(float(a))
        X = Fraction(2) ** (c - 127)
        assert 4 * X <= Fraction(float(a)) < 8 * X, (float(a), c)
    assert oracle_mod.mx_scale_code(0.0) == 0


def test_mx_elements_are_the_nearest_grid_points(oracle_mod):
    """Every dequantized element is the nearest E2M1 value (ties to even) of x / X,
    checked in exact rational arithmetic."""
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((6, 64)) * np.exp(rng.uniform(-8, 8, (6, 1)))).astype(np.float32)
    x[0, :8] = [0.0, -0.0, 1e-30, -1e-30, 2.5, -3.5, 5.0, 0.75]       # ties and tiny values
    q = oracle_mod.mx_quantize(x)
    d = oracle_mod.mx_dequant(q)
    for i in range(x.shape[0]):
        for b in range(2):
            X = Fraction(2) ** (int(q["scales"][i, b]) - 127)
            for j in range(32 * b, 32 * b + 32):
                y = Fraction(float(np.float32(Fraction(float(x[i, j])) / X)))   # one fp32 rounding
                assert Fraction(d[i, j]) == _brute_e2m1_times(y) * X, (i, j, float(x[i, j]))


def test_mx_round_trip_and_saturation(oracle_mod):
    """Blocks of E2M1 values times 2^k that contain +-6 * 2^k come back exactly; a block
    maximum of 7 * 2^k saturates to 6 * 2^k."""
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], np.float32)
    rng = np.random.default_rng(13)
    for k in (-20, -3, 0, 5, 30):
        v = rng.choice(grid, 32) * rng.choice([-1, 1], 32)
        v[7] = 6.0
        x = (v * np.float32(2.0 ** k)).astype(np.float32)[None, :]
        q = oracle_mod.mx_quantize(x)
        assert np.array_equal(oracle_mod.mx_dequant(q)[0], x[0].astype(np.float64)), k
        x2 = x.copy()
        x2[0, 7] = np.float32(7.0 * 2.0 ** k)
        d2 = oracle_mod.mx_dequant(oracle_mod.mx_quantize(x2))[0]
        assert d2[7] == 6.0 * 2.0 ** k


def test_mx_col_operand_is_the_transpose(oracle_mod):
    x = np.random.default_rng(14).standard_normal((64, 96)).astype(np.float32)
    a = oracle_mod.mx_quantize(x, col=True)
    b = oracle_mod.mx_quantize(np.ascontiguousarray(x.T))
    assert np.array_equal(a["codes"], b["codes"]) and np.array_equal(a["scales"], b["scales"])


def test_nvfp4_error_below_mxfp4_on_heavy_tailed_activations(oracle_mod):
    """The direction of the page's format comparison at the quantizer level (no training):
    on the heavy-tailed activations (Student-t(3), 1% of channels x50) the oracle's NVFP4
    (1x16, E4M3 scales, FP32 tensor scale) dequantizes closer to the input than its MXFP4
    (1x32, power-of-two scales); likewise on N(0, 1) data."""
    import torch
    from nvfp4_bit_quantized_gb300 import inputs
    X = inputs.student_t((128, 512), 3, seed=3)
    inputs.outlier_columns(X, 0.01, 50.0, seed=103)
    bits = X.contiguous().view(torch.int16).numpy().view(np.uint16)
    x = X.float().numpy().astype(np.float64)

    def rel(d):
        return float(np.linalg.norm(d - x) / np.linalg.norm(x))
    e_nv = rel(oracle_mod.dequant(oracle_mod.quantize(bits, oracle_mod.ROW)))
    e_mx = rel(oracle_mod.mx_dequant(oracle_mod.mx_quantize(bits)))
    assert 0 < e_nv < e_mx, (e_nv, e_mx)
    # the same inputs on a N(0, 1) tensor: the ordering does not hinge on the outliers
    Y = inputs.normal((128, 512), 1.0, seed=4)
    ybits = Y.contiguous().view(torch.int16).numpy().view(np.uint16)
    y = Y.float().numpy().astype(np.float64)
    e_nv_y = float(np.linalg.norm(oracle_mod.dequant(oracle_mod.quantize(ybits, oracle_mod.ROW)) - y) / np.linalg.norm(y))
    e_mx_y = float(np.linalg.norm(oracle_mod.mx_dequant(oracle_mod.mx_quantize(ybits)) - y) / np.linalg.norm(y))
    assert e_nv_y < e_mx_y, (e_nv_y, e_mx_y)
