"""Host-side checks of arithmetic the CUDA kernels rely on, emulated exactly.

The restore kernel divides the exact fp32 sum of three E4M3 references by 3 (the
reference mean of a token with k_i = 3, ResidualKV notes §2.2) without a division
instruction: q = RN(s * c) with c = RN(1/3), r = RN(s - 3 q) (one fused multiply-add,
exact here), then RN(q + r * c) (one fused multiply-add).  This is the residual
correction of a reciprocal product (Markstein's method for correctly rounded division,
with the quotient refined once by its residual).  The test emulates the three roundings
exactly and checks, for every sum of three finite E4M3 values, that the result is the
correctly rounded quotient RN(s / 3)."""
from fractions import Fraction

import numpy as np


def _e4m3_finite():
    """All finite E4M3 values (OCP 'e4m3fn': bias 7, three mantissa bits, subnormals at
    exponent field 0, S.1111.111 is NaN), as exact binary64 numbers."""
    vals = []
    for b in range(256):
        s, e, m = b >> 7, (b >> 3) & 15, b & 7
        if e == 15 and m == 7:
            continue
        x = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        vals.append(-x if s else x)
    return np.unique(np.array(vals))


def _rn32_exact(x: Fraction) -> Fraction:
    """Round a rational to the nearest binary32 value, ties to even (no overflow here)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                     # subnormals share the smallest exponent
    scale = Fraction(2) ** (23 - e)      # ulp = 2^(e - 23)
    y = a * scale
    n = y.numerator // y.denominator
    rem = y - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n / scale


def test_div3_residual_correction_is_correctly_rounded_for_all_e4m3_triple_sums():
    v = _e4m3_finite()
    sums = np.unique((v[:, None, None] + v[None, :, None] + v[None, None, :]).ravel())
    # every such sum is a multiple of 2^-9 below 3 * 448 in magnitude: exact in binary32,
    # which is how the kernel holds it
    assert np.all(sums.astype(np.float32).astype(np.float64) == sums)
    assert len(sums) == 256317
    c = Fraction(0x3EAAAAAB & 0x7FFFFF | 0x800000, 2 ** 25)          # RN(1/3) = 0x3EAAAAAB
    assert c == _rn32_exact(Fraction(1, 3))
    si = np.round(sums * 512).astype(np.int64)                       # s = si / 512 exactly
    bad = []
    for k in si.tolist():
        s = Fraction(k, 512)
        q = _rn32_exact(s * c)
        r = _rn32_exact(s - 3 * q)
        got = _rn32_exact(q + r * c)
        if got != _rn32_exact(s / 3):
            bad.append(k)
    assert not bad, f"{len(bad)} sums not correctly rounded, e.g. {bad[:3]}"


def test_div3_plain_reciprocal_product_is_not_enough():
    """Negative control: without the residual step, RN(s * RN(1/3)) misses the correctly
    rounded quotient for some of the same sums (so the check above can fail)."""
    c = Fraction(0x3EAAAAAB & 0x7FFFFF | 0x800000, 2 ** 25)
    misses = 0
    for k in range(1, 4096):
        s = Fraction(k, 512)
        misses += _rn32_exact(s * c) != _rn32_exact(s / 3)
    assert misses > 0
