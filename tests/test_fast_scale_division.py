"""The fused quant kernel forms the block scale RN(amax / 448) without a division: amax is a
bf16 value, and for every such value in [2^-100, max finite] Markstein's correction
q0 = RN(amax * c), r = amax - 448 * q0 (exact), RN(q0 + r * c) with c = RN(1/448) gives the
correctly rounded quotient (P. Markstein, IBM J. Res. Dev. 34(1), 1990).  This test re-checks
that claim exhaustively with exact rational arithmetic (no GPU, no product code)."""
import math
import struct
from fractions import Fraction as F


def rn32(q: F) -> F:
    """Round-to-nearest-even of a rational to binary32 (normal range, either sign)."""
    if q == 0:
        return F(0)
    sign = -1 if q < 0 else 1
    q = abs(q)
    e = q.numerator.bit_length() - q.denominator.bit_length()
    while F(2) ** e > q:
        e -= 1
    while F(2) ** (e + 1) <= q:
        e += 1
    ulp = F(2) ** (e - 23)
    m = q / ulp
    fl = math.floor(m)
    rem = m - fl
    if rem > F(1, 2) or (rem == F(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * ulp


def bf16_value(bits: int) -> F:
    return F(struct.unpack("<f", struct.pack("<I", bits << 16))[0])


def test_rn32_helper_against_float32_rounding():
    import numpy as np
    rng = np.random.default_rng(0)
    for v in rng.standard_normal(200) * 1e3:
        assert rn32(F(float(v))) == F(float(np.float32(v)))


def test_markstein_scale_is_correctly_rounded_for_every_bf16_amax():
    c = rn32(F(1, 448))
    assert c == F(float(struct.unpack("<f", struct.pack("<f", 1.0 / 448.0))[0]))
    checked = 0
    for bits in range(0x0080, 0x7F80):  # positive normal, finite bf16
        a = bf16_value(bits)
        if a < F(2) ** -100:
            continue
        q0 = rn32(a * c)
        r = a - 448 * q0
        assert rn32(r) == r, hex(bits)          # the FMA residual is exact
        assert rn32(q0 + r * c) == rn32(a / 448), hex(bits)
        checked += 1
    assert checked == 29184
