"""Pins for oracle.formats: codebooks, E4M3 decode, global inversion, BF16 rounding.

Each check compares the oracle with something other than itself: hand-derived
worked values (tests/golden), the formats' bit-field definitions evaluated in
exact rational arithmetic (tests/exact.py), or library routines (torch's
float8_e4m3fn and float32->bfloat16 casts).
"""

import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats
from tests.exact import (bf16_exact, bf16_round_exact, e2m1_exact, e4m3_exact, f16_exact, f16_round_exact,
                         swizzle_scales_by_tiles)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_kv(name):
    out = {}
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                k, v = line.split(":", 1)
                out[k.strip()] = v.split()
            else:
                rows.append(line.split())
    return out, rows


def test_e2m1_worked_row():
    kv, _ = _read_kv("e2m1_worked_row.txt")
    packed = np.array([int(b, 16) for b in kv["bytes"]], dtype=np.uint8)
    codes = np.empty(16, dtype=np.int64)
    codes[0::2] = packed & 0xF
    codes[1::2] = packed >> 4
    got = formats.e2m1_value(codes)
    want = np.array([float(v) for v in kv["values"]])
    assert np.array_equal(got, want)
    assert np.array_equal(np.signbit(got), np.signbit(want))   # code 8 is -0.0


def test_e2m1_matches_bit_fields():
    for c in range(16):
        v = formats.e2m1_value(c)
        assert Fraction(float(v)) == e2m1_exact(c)
    assert np.signbit(formats.e2m1_value(8))


def test_e4m3_worked_values():
    _, rows = _read_kv("e4m3_worked.txt")
    for code, val in rows:
        got = float(formats.e4m3_value(int(code, 16)))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val)
            assert math.copysign(1, got) == math.copysign(1, float(val))


def test_e4m3_all_codes_against_torch_and_bit_fields():
    codes = np.arange(256)
    ours = formats.e4m3_value(codes)
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2                                      # 0x7F and 0xFF
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    for c in range(256):
        ex = e4m3_exact(c)
        if ex is None:
            assert math.isnan(ours[c])
        else:
            assert Fraction(float(ours[c])) == ex
    assert ours[0x7E] == 448.0 and np.nanmax(ours) == 448.0


def test_global_inversion_worked_value():
    kv, _ = _read_kv("divisor_inversion.txt")
    d = float(kv["divisor"][0])
    g = formats.global_multiplier(d, True)
    assert g.dtype == np.float32
    assert struct.unpack("<I", struct.pack("<f", float(g)))[0] == int(kv["g_bits"][0], 16)
    # without the divisor flag the stored value is used as is
    assert formats.global_multiplier(d, False) == np.float32(448.0)
    # the IEEE float32 quotient is the correctly rounded reciprocal
    for dv in (448.0, 3.0, 24366.764, 1e-3, 7.0e5):
        got = Fraction(float(formats.global_multiplier(dv, True)))
        exact = 1 / Fraction(float(np.float32(dv)))
        # nearest float32: the neighbours one ulp away are not closer
        ulp = Fraction(2) ** (math.frexp(float(got))[1] - 24)
        assert abs(got - exact) <= ulp / 2


def test_bf16_rounding_matches_torch_on_float32():
    r = np.random.default_rng(7)
    bits = r.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    # add hand-picked edges: ties, max finite, overflow boundary, subnormals, zeros
    edges = np.array([0x3F808000, 0x3F818000, 0x3F80FFFF, 0x7F7F7FFF, 0x7F7F8000,
                      0x7F7FFFFF, 0x00008000, 0x00018000, 0x0000FFFF, 0x80000000,
                      0x00000001, 0x807FFFFF, 0x7F800000, 0xFF800000], dtype=np.uint32)
    bits = np.concatenate([bits, edges])
    f = bits.view(np.float32)
    finite = np.isfinite(f)
    f = f[finite]
    ours = formats.bf16_bits(f.astype(np.float64))
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_rounding_is_single_rounding():
    # 1 + 2^-8 + 2^-30 is above the BF16 tie between 1 and 1 + 2^-7; rounding it to
    # float32 first would land exactly on the tie and then go to the even neighbour 1.0.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert int(formats.bf16_bits(v)) == 0x3F81
    assert int(formats.bf16_bits(np.float32(v))) == 0x3F80       # the double-rounded result
    for x in (1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8) - 2.0 ** -40,
              2.0 ** -130 * 1.5, 2.0 ** -133 / 2, 2.0 ** -133 * 0.75, 3.3e38, 3.4e38,
              -0.0, 0.0, 2.0 ** 127 * 1.99609375):
        want = bf16_round_exact(Fraction(x), negative_zero=math.copysign(1, x) < 0)
        assert int(formats.bf16_bits(x)) == want, hex(want)


def test_bf16_rounding_against_exact_rationals_random():
    r = np.random.default_rng(11)
    mant = r.integers(1, 2 ** 52, size=3000)
    exps = r.integers(-140, 128, size=3000)
    vals = np.ldexp(1.0 + mant / 2.0 ** 52, exps)
    ours = formats.bf16_bits(vals)
    for v, b in zip(vals, ours):
        assert int(b) == bf16_round_exact(Fraction(float(v)))


def test_bf16_specials_and_roundtrip():
    assert int(formats.bf16_bits(np.nan)) & 0x7FFF == 0x7FC0
    assert int(formats.bf16_bits(-np.inf)) == 0xFF80
    assert int(formats.bf16_bits(np.inf)) == 0x7F80
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = formats.bf16_to_float(allbits)
    finite = np.isfinite(vals)
    assert np.array_equal(formats.bf16_bits(vals[finite]), allbits[finite])
    for b in (0x0001, 0x3F80, 0x7F7F, 0x8080, 0xC0C0):
        assert Fraction(float(formats.bf16_to_float(np.uint16(b)))) == bf16_exact(b)


def test_plant_wrong_tie_rule_is_caught(monkeypatch):
    """A planted mistake (ties away from zero) must fail the rounding pins."""
    def bad(values):
        v = np.asarray(values, dtype=np.float64)
        a = np.abs(v)
        _, e = np.frexp(a)
        q = np.where(a >= 2.0 ** -126, e - 8, -133)
        r = np.floor(np.ldexp(a, -q) + 0.5)
        f32 = (np.ldexp(r, q) * np.sign(v)).astype(np.float32)
        return (f32.view(np.uint32) >> 16).astype(np.uint16)
    monkeypatch.setattr(formats, "bf16_bits", bad)
    with pytest.raises(AssertionError):
        test_bf16_rounding_is_single_rounding()


# ---------------------------------------------------------------- FP16 ---
def test_f16_rounding_matches_torch_on_float32():
    r = np.random.default_rng(17)
    n = 200000
    mant = r.integers(0, 2 ** 23, size=n)
    exps = r.integers(-30, 18, size=n)            # subnormal range, normal range, overflow
    sgn = np.where(r.integers(0, 2, size=n) == 1, -1.0, 1.0)
    f = (sgn * np.ldexp(1.0 + mant / 2.0 ** 23, exps)).astype(np.float32)
    edges = np.array([65504.0, 65519.99, 65520.0, 65536.0, 2.0 ** -24, 2.0 ** -25, 1.5 * 2.0 ** -25,
                      2.0 ** -14 - 2.0 ** -26, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, -0.0, 0.0,
                      3.0e38, -65520.0], dtype=np.float32)
    f = np.concatenate([f, edges])
    ours = formats.f16_bits(f.astype(np.float64))
    ref = torch.from_numpy(f.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f16_rounding_is_single_rounding():
    # 1 + 2^-11 + 2^-40 lies above the FP16 tie between 1 and 1 + 2^-10; rounding it to
    # float32 first lands exactly on the tie, which then goes to the even neighbour 1.0.
    v = 1.0 + 2.0 ** -11 + 2.0 ** -40
    assert int(formats.f16_bits(v)) == 0x3C01
    assert int(formats.f16_bits(np.float32(v))) == 0x3C00       # the double-rounded result
    for x in (1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, -(1.0 + 2.0 ** -11) - 2.0 ** -45,
              2.0 ** -20 * 1.5, 2.0 ** -24 / 2, 2.0 ** -24 * 0.75, 65504.0, 65519.999, 65520.0,
              -0.0, 0.0, 2.0 ** -14 * (1 - 2.0 ** -12)):
        want = f16_round_exact(Fraction(x), negative_zero=math.copysign(1, x) < 0)
        assert int(formats.f16_bits(x)) == want, (x, hex(want))


def test_f16_rounding_against_exact_rationals_random():
    r = np.random.default_rng(13)
    mant = r.integers(1, 2 ** 52, size=3000)
    exps = r.integers(-30, 18, size=3000)
    vals = np.ldexp(1.0 + mant / 2.0 ** 52, exps)
    ours = formats.f16_bits(vals)
    for v, b in zip(vals, ours):
        assert int(b) == f16_round_exact(Fraction(float(v)))


def test_f16_specials_and_roundtrip():
    assert int(formats.f16_bits(np.nan)) & 0x7FFF == 0x7E00
    assert int(formats.f16_bits(-np.inf)) == 0xFC00
    assert int(formats.f16_bits(np.inf)) == 0x7C00
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = formats.f16_to_float(allbits)
    finite = np.isfinite(vals)
    assert np.array_equal(formats.f16_bits(vals[finite]), allbits[finite])
    for b in (0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0x8400, 0xC0C0):
        assert Fraction(float(formats.f16_to_float(np.uint16(b)))) == f16_exact(b)


def test_plant_f16_wrong_tie_rule_is_caught(monkeypatch):
    """Ties away from zero instead of to even must fail the FP16 rounding pins."""
    def bad(values):
        v = np.asarray(values, dtype=np.float64)
        a = np.abs(v)
        _, e = np.frexp(a)
        q = np.where(a >= 2.0 ** -14, e - 11, -24)
        r = np.floor(np.ldexp(a, -q) + 0.5)
        return (np.ldexp(r, q) * np.sign(v)).astype(np.float16).view(np.uint16)
    monkeypatch.setattr(formats, "f16_bits", bad)
    with pytest.raises(AssertionError):
        test_f16_rounding_is_single_rounding()


# ----------------------------------------------------- swizzled scales ---
def test_swizzled_offsets_worked_values():
    rows = []
    with open(os.path.join(os.path.dirname(__file__), "golden", "swizzled_scale_offsets.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(v) for v in line.split()])
    for n, j, off in rows:
        assert int(formats.swizzled_scale_offset(n, j, 12)) == off, (n, j)


@pytest.mark.parametrize("N,K", [(1, 16), (128, 64), (300, 192), (257, 2064)])
def test_unswizzle_inverts_the_tile_walk(N, K):
    r = np.random.default_rng(N + K)
    lin = r.integers(0, 256, size=(N, K // 16), dtype=np.uint8)
    sw = swizzle_scales_by_tiles(lin, N, K)
    assert sw.size == formats.swizzled_scales_size(N, K)
    assert np.array_equal(formats.unswizzle_scales(sw, N, K), lin)
    # every (n, j) lands on a distinct byte
    offs = formats.swizzled_scale_offset(np.arange(N)[:, None], np.arange(K // 16)[None, :], K // 16)
    assert np.unique(offs).size == offs.size
