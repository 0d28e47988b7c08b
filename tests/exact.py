"""Exact rational arithmetic used to pin the oracle (tests only).

Everything here is derived from the bit-level definitions of the formats and
computed with ``fractions.Fraction``, so it shares no arithmetic with the
float64 oracle: decoding reads exponent/mantissa fields (not a codebook
table), and BF16 rounding compares exact remainders against one half.
"""

from fractions import Fraction

import numpy as np


def e2m1_exact(code):
    """E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        mag = Fraction(m, 2)                      # subnormal: m * 2**(1-1) * 1/2
    else:
        mag = Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
    return -mag if s else mag


def e4m3_exact(code):
    """float8_e4m3fn: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits.

    Returns None for the NaN patterns (exponent 15, mantissa 7)."""
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 7
    if e == 15 and m == 7:
        return None
    if e == 0:
        mag = Fraction(m, 8) * Fraction(1, 2 ** 6)
    else:
        mag = (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -mag if s else mag


def f32_exact(x):
    return Fraction(float(np.float32(x)))


def _floor_log2(q):
    """floor(log2(q)) for a positive Fraction."""
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    if Fraction(2) ** (e + 1) <= q:
        e += 1
    return e


def bf16_round_exact(v, negative_zero=False):
    """Round a Fraction to BF16 (nearest, ties to even); returns the 16-bit pattern."""
    if v == 0:
        return 0x8000 if negative_zero else 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = max(_floor_log2(a), -126)
    quantum = Fraction(2) ** (e - 7)
    q = a / quantum
    m = q.numerator // q.denominator
    rem = q - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and (m & 1)):
        m += 1
    # m is now the integer significand in units of the quantum (<= 256)
    if m == 256:
        m = 128
        e += 1
    if m < 128:                                   # subnormal (only when e == -126)
        return sign | m
    exp_field = e + 127
    if exp_field >= 255:
        return sign | 0x7F80
    return sign | (exp_field << 7) | (m - 128)


def bf16_exact(bits):
    """Exact value of a finite BF16 pattern."""
    s = (bits >> 15) & 1
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    if e == 0:
        mag = Fraction(f, 128) * Fraction(2) ** -126
    else:
        mag = (1 + Fraction(f, 128)) * Fraction(2) ** (e - 127)
    return -mag if s else mag


def f16_round_exact(v, negative_zero=False):
    """Round a Fraction to FP16 (IEEE binary16, nearest, ties to even); returns
    the 16-bit pattern.  1 sign bit, 5 exponent bits (bias 15), 10 fraction bits."""
    if v == 0:
        return 0x8000 if negative_zero else 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = max(_floor_log2(a), -14)
    quantum = Fraction(2) ** (e - 10)
    q = a / quantum
    m = q.numerator // q.denominator
    rem = q - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and (m & 1)):
        m += 1
    if m == 2048:
        m = 1024
        e += 1
    if m < 1024:                                  # subnormal (only when e == -14)
        return sign | m
    exp_field = e + 15
    if exp_field >= 31:
        return sign | 0x7C00
    return sign | (exp_field << 10) | (m - 1024)


def f16_exact(bits):
    """Exact value of a finite FP16 pattern."""
    s = (bits >> 15) & 1
    e = (bits >> 10) & 0x1F
    f = bits & 0x3FF
    if e == 0:
        mag = Fraction(f, 1024) * Fraction(2) ** -14
    else:
        mag = (1 + Fraction(f, 1024)) * Fraction(2) ** (e - 15)
    return -mag if s else mag


def swizzle_scales_by_tiles(lin, N, K):
    """Independent construction: walk the 128 x 4 tiles and the 32 x (4 x 4)
    interleave inside each, writing bytes in storage order."""
    G = K // 16
    Np, Gp = -(-N // 128) * 128, -(-G // 4) * 4
    pad = np.zeros((Np, Gp), dtype=np.uint8)
    pad[:N, :G] = lin
    out = []
    for rt in range(Np // 128):
        for ct in range(Gp // 4):
            for r32 in range(32):
                for quarter in range(4):
                    for c in range(4):
                        out.append(pad[rt * 128 + quarter * 32 + r32, ct * 4 + c])
    return np.array(out, dtype=np.uint8)
