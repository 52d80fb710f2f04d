"""Division by 6 in the block-scale computation, checked exactly on the host.

The encoders compute S_b = e4m3(RN(amax_b / 6) * s_enc) (NVIDIA's NVFP4 pretraining
page, the block-scale step of the quantization recipe).  Instead of the general IEEE
division they use the correction step q0 = RN(a * RN(1/6)), r = a - 6 q0 (exact, one
fma), q = RN(q0 + r * RN(1/6)) (Markstein 1990; Brisebarre, Muller and Raina 2004),
falling back to the division when a < 6 * 2^-126.  This test replays that step with
IEEE binary32 arithmetic on every bf16 value and every fp32 significand and compares
it with the correctly rounded quotient.

Why the emulation is exact: numpy's float32 multiply rounds to nearest like
__fmul_rn; the remainder a - 6 q0 needs at most 27 bits and is exact in float64
(the device fma computes it exactly too); q0 + r * RN(1/6) spans fewer than 53 bits
(|r| is a few units of q0's last place), so float64 holds it exactly and the one
rounding to float32 is the fma's.  The reference a / 6 in float64 rounded to float32
is the correctly rounded quotient: n / 3 for integer n not divisible by 3 stays more
than 2^-53 (relative) away from every 25-bit dyadic midpoint.
"""
import numpy as np

INV6 = np.array([0x3E2AAAAB], dtype=np.uint32).view(np.float32)[0]
THRESHOLD = np.float32(6 * 2.0 ** -126)


def correction(a):
    a = np.asarray(a, dtype=np.float32)
    q0 = (a * INV6).astype(np.float32)
    r = a.astype(np.float64) - q0.astype(np.float64) * 6.0
    return (r * np.float64(INV6) + q0.astype(np.float64)).astype(np.float32)


def rn_div6(a):
    return (np.asarray(a, dtype=np.float32).astype(np.float64) / 6.0).astype(np.float32)


def test_inverse_constant_is_rn_one_sixth():
    from fractions import Fraction
    err = abs(Fraction(float(INV6)) - Fraction(1, 6))
    ulp = Fraction(2) ** (-3 - 23)          # 1/6 lies in [2^-3, 2^-2)
    assert err <= ulp / 2


def test_every_positive_finite_bf16():
    bits = np.arange(1, 0x7F80, dtype=np.uint32) << 16
    a = bits.view(np.float32)
    assert np.array_equal(correction(a).view(np.uint32), rn_div6(a).view(np.uint32))


def test_every_fp32_significand_normal_quotient():
    # The step commutes with scaling by powers of two while nothing is subnormal, so
    # one full binade of significands stands for all of them; the bottom binades
    # (where q0 is near the subnormal boundary) and the top binade (near FLT_MAX) are
    # swept in full as well.
    exps = [1, 2, 3, 4, 5, 127, 128, 200, 253, 254]
    sig = np.arange(0, 1 << 23, dtype=np.uint32)
    for e in exps:
        a = ((np.uint32(e) << 23) | sig).view(np.float32)
        a = a[a >= THRESHOLD]
        got, ref = correction(a), rn_div6(a)
        assert np.isfinite(got).all()
        bad = np.nonzero(got.view(np.uint32) != ref.view(np.uint32))[0]
        assert bad.size == 0, (e, a[bad[:4]])


def test_subnormal_quotients_need_the_fallback():
    # Below 6 * 2^-126 the quotient is subnormal and the step misses by one unit for
    # some inputs: the device falls back to the IEEE division there.
    a = np.arange(1, 0x00C00000, dtype=np.uint32).view(np.float32)
    a = a[a < THRESHOLD]
    mism = np.count_nonzero(correction(a).view(np.uint32) != rn_div6(a).view(np.uint32))
    assert mism > 0
