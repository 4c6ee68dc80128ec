"""Exactness of the fused FP8 dispatch's quotient forms, proved on the host.

The OCP E4M3 quantisation of the MORI-EP dispatch ("EPv2 configuration and
lifecycle": one fp32 scale per 128 elements) needs scale = fl32(a / 448) for a
block maximum a, and fl32(x / scale) per element.  The CUDA kernel forms both
as a product with a rounded reciprocal plus one FMA correction (Markstein's
division step).  These tests check, with exact rational arithmetic and no GPU,
that the scale form equals the IEEE quotient for every value a block maximum
can take (every finite non-negative bf16), and that the negated-residual form
of the element quotient keeps the sign of a zero input.  The GPU test of the
codes themselves (every bf16 x under many block maxima) is in
test_gpu_fp8_codes.py.
"""
from fractions import Fraction

import numpy as np


def _rn32(x: Fraction) -> Fraction:
    """Round a rational to the nearest binary32 value, ties to even
    (subnormals included; the inputs here never overflow)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    ax = abs(x)
    e = ax.numerator.bit_length() - ax.denominator.bit_length()
    while Fraction(2) ** e > ax:
        e -= 1
    while Fraction(2) ** (e + 1) <= ax:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 23)
    n = ax / quantum
    whole = n.numerator // n.denominator
    rest = n - whole
    if rest > Fraction(1, 2) or (rest == Fraction(1, 2) and whole % 2 == 1):
        whole += 1
    return sign * whole * quantum


def _bf16(bits: int) -> Fraction:
    return Fraction(float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0]))


def test_rn32_agrees_with_numpy_rounding():
    # the helper itself, against numpy's float64 -> float32 conversion on
    # values a float64 holds exactly (normal, subnormal, ties)
    rng = np.random.default_rng(5)
    for v in np.concatenate([rng.standard_normal(2000) * 1e3,
                             rng.standard_normal(200) * 1e-40,
                             [1 + 2.0 ** -24, 1 + 3 * 2.0 ** -24, 2.0 ** -149 * 1.5]]):
        assert float(_rn32(Fraction(float(v)))) == float(np.float32(v))


def test_block_scale_reciprocal_form_equals_the_quotient_for_every_bf16_maximum():
    inv = _rn32(Fraction(1, 448))
    assert float(inv) == float(np.float32(1) / np.float32(448))
    plain_misses = 0
    for bits in range(0, 0x7F80):            # +0 .. the largest finite bf16
        a = _bf16(bits)
        exact = _rn32(a / 448)
        q0 = _rn32(a * inv)                  # RN(a * RN(1/448))
        e = _rn32(a - q0 * 448)              # fma(-q0, 448, a)
        assert _rn32(q0 + e * inv) == exact, hex(bits)   # fma(e, RN(1/448), q0)
        plain_misses += q0 != exact
    # the correction matters: the bare product misses about half the values
    assert plain_misses > 10000


def test_negated_residual_keeps_the_sign_of_zero():
    f = np.float32
    for scale in (f(2.0 ** -90), f(1 / 448), f(3.5), f(1e30)):
        r = f(1) / scale
        for x in (f(0.0), f(-0.0)):
            q0 = x * r
            nres = q0 * scale + (-x)          # fma(q0, scale, -x): exact on zeros
            q = nres * (-r) + q0              # fma(nres, -r, q0)
            assert q == 0 and np.signbit(q) == np.signbit(x)
