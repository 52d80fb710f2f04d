"""The device codecs the kernels use, pinned element by element to the oracle.
(Diagnostic entry points run the exact device routines.)"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_bit_quantized_gb300 import _lib
    return _lib


def _s():
    return torch.cuda.current_stream().cuda_stream


def test_e4m3_cast_matches_oracle_dense_sweep(L, oracle_mod):
    # every fp32 in [0, 1024] with the low 8 mantissa bits stepped by 1 (plus subnormal range)
    u = np.arange(0, 0x44800000 >> 8, dtype=np.uint64) << 8
    v = u.astype(np.uint32).view(np.float32)
    v = np.concatenate([v, np.array([448, 464, 465, 1e9, 2.0 ** -10, 2.0 ** -11, 0.0], np.float32)])
    got = torch.empty(v.size, dtype=torch.uint8, device="cuda")
    vt = torch.from_numpy(v).cuda()
    L.check(L.lib().nvfp4_debug_e4m3(vt.data_ptr(), v.size, got.data_ptr(), _s()))
    ref = oracle_mod.e4m3_encode(v)
    bad = np.nonzero(got.cpu().numpy() != ref)[0]
    assert bad.size == 0, [(float(v[i]), int(got[i]), int(ref[i])) for i in bad[:10]]


def _e2m1_sweep():
    rng = np.random.default_rng(0)
    grid = [0, .5, 1, 1.5, 2, 3, 4, 6]
    pts = []
    for a, b in zip(grid[:-1], grid[1:]):
        m = np.float32((a + b) / 2)
        pts += [a, b, m, np.nextafter(m, np.float32(0)), np.nextafter(m, np.float32(9))]
    pts += [0.0, 6.0, 6.5, 1e30, 1e-30, 1e-45]
    v = np.array(pts, np.float32)
    v = np.concatenate([v, -v, rng.uniform(-8, 8, 200000).astype(np.float32),
                        (rng.standard_normal(50000) * 1e-3).astype(np.float32)])
    return v


@pytest.mark.parametrize("hw", [0, 1])
def test_e2m1_rne_matches_oracle(L, oracle_mod, hw):
    """hw=0: the software threshold rule; hw=1: the cvt.rn.satfinite.e2m1x2
    instruction the kernels use.  Both must equal the oracle's RNE reading
    (ties to even, saturation, the sign kept on zero)."""
    y = _e2m1_sweep()
    yt = torch.from_numpy(y).cuda()
    got = torch.empty(y.size, dtype=torch.uint8, device="cuda")
    L.check(L.lib().nvfp4_debug_e2m1(yt.data_ptr(), None, y.size, L.RNE, hw, got.data_ptr(), _s()))
    ref = oracle_mod.e2m1_encode_rne(y)
    g = got.cpu().numpy()
    bad = np.nonzero(g != ref)[0]
    assert bad.size == 0, [(float(y[i]), int(g[i]), int(ref[i])) for i in bad[:10]]

def test_e2m1_sr_matches_oracle(L, oracle_mod):
    y = _e2m1_sweep()
    r = np.random.default_rng(1).integers(0, 65536, y.size).astype(np.uint32)
    r[:16] = [0, 1, 32767, 32768, 65535, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12]
    yt, rt = torch.from_numpy(y).cuda(), torch.from_numpy(r.view(np.int32)).cuda()
    got = torch.empty(y.size, dtype=torch.uint8, device="cuda")
    L.check(L.lib().nvfp4_debug_e2m1(yt.data_ptr(), rt.data_ptr(), y.size, L.SR, 0, got.data_ptr(), _s()))
    ref = oracle_mod.e2m1_encode_sr(y, r)
    assert np.array_equal(got.cpu().numpy(), ref)


def test_philox_matches_oracle(L, oracle_mod):
    rng = np.random.default_rng(2)
    n = 4096
    ctr = rng.integers(0, 2 ** 32, (n, 4), dtype=np.uint64).astype(np.uint32)
    ctr[0] = 0
    for key in (0, 1, 0xDEADBEEFCAFEF00D):
        ct = torch.from_numpy(ctr.view(np.int32)).cuda()
        out = torch.empty((n, 4), dtype=torch.int32, device="cuda")
        L.check(L.lib().nvfp4_debug_philox(ct.data_ptr(), n, key, out.data_ptr(), _s()))
        got = out.cpu().numpy().view(np.uint32)
        for i in range(0, n, 97):
            assert np.array_equal(got[i], oracle_mod.philox4x32_10(ctr[i], [key & 0xFFFFFFFF, key >> 32]))
