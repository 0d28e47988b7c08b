"""Pins for oracle.dense: dequantization, AWQ scaling and the GEMM.

Independent of the oracle: hand-derived worked values (tests/golden), exact
rational arithmetic from the formats' bit fields (tests/exact.py), pure-Python
brute-force dot products, and invariants (dequant(quant(x)) idempotence, the
power-of-two exact case).  Planted mistakes (a skipped divisor inversion, a
swapped nibble order, a dropped AWQ scale) must be caught.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import dense, formats
from tests.exact import bf16_exact, bf16_round_exact, e2m1_exact, e4m3_exact, f16_exact, f16_round_exact, f32_exact
from w4a16_nvfp4_weight_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    kv, rows = {}, []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                k, v = line.split(":", 1)
                kv[k.strip()] = v.split()
            else:
                rows.append(line.split())
    return kv, rows


def _pack(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def _exact_dequant(code, scale_code, g, act="bf16"):
    s = e4m3_exact(scale_code)
    v = e2m1_exact(code) * s * f32_exact(g)
    neg_zero = v == 0 and (((code >> 3) ^ (scale_code >> 7)) & 1) == 1
    rnd = bf16_round_exact if act == "bf16" else f16_round_exact
    return rnd(v, negative_zero=neg_zero)


def test_worked_row_with_unit_scales():
    kv, _ = _golden_rows("e2m1_worked_row.txt")
    packed = np.array([[int(b, 16) for b in kv["bytes"]]], dtype=np.uint8)
    scales = np.array([[0x38]], dtype=np.uint8)
    w = dense.dequant(packed, scales, 1.0, False, 16)
    assert [f"{int(b):04X}" for b in w[0]] == kv["bf16"]
    # X = ones: the row sums to exactly zero
    x = np.full((1, 16), 0x3F80, dtype=np.uint16)
    y, yb = dense.linear(x, packed, scales, 1.0, False)
    assert y[0, 0] == 0.0 and int(yb[0, 0]) & 0x7FFF == 0


def test_divisor_inversion_worked_values():
    kv, rows = _golden_rows("divisor_inversion.txt")
    d = float(kv["divisor"][0])
    for code, sc, want in rows:
        c, s = int(code, 16), int(sc, 16)
        codes = np.zeros((1, 16), dtype=np.uint8)
        codes[0, 0] = c
        w = dense.dequant(_pack(codes), np.array([[s]], dtype=np.uint8), d, True, 16)
        assert f"{int(w[0, 0]):04X}" == want


def test_planted_skipped_inversion_is_caught(monkeypatch):
    monkeypatch.setattr(dense, "global_multiplier", lambda v, is_div: np.float32(v))
    with pytest.raises(AssertionError):
        test_divisor_inversion_worked_values()


def test_planted_nibble_swap_is_caught(monkeypatch):
    def swapped(packed, K):
        p = np.asarray(packed, dtype=np.uint8)
        codes = np.empty((p.shape[0], K), dtype=np.int64)
        codes[:, 0::2] = p >> 4
        codes[:, 1::2] = p & 0xF
        return codes
    monkeypatch.setattr(dense, "unpack_codes", swapped)
    with pytest.raises(AssertionError):
        test_worked_row_with_unit_scales()


@pytest.mark.parametrize("divisor", [448.0, 3.0, 24366.764, 0.37, 1.0e-30])
def test_dequant_exact_over_all_codes_and_scales(divisor):
    """Every (code, scale) pair against exact rational rounding (single rounding)."""
    codes = np.tile(np.arange(16, dtype=np.uint8), (256, 1))          # [256, 16]
    scales = np.arange(256, dtype=np.uint8).reshape(256, 1)
    w = dense.dequant(_pack(codes), scales, divisor, True, 16)
    g = formats.global_multiplier(divisor, True)
    for s in range(256):
        for c in range(16):
            got = int(w[s, c])
            if e4m3_exact(s) is None:
                assert got & 0x7FFF == 0x7FC0
                assert (got >> 15) == (((c >> 3) ^ (s >> 7)) & 1)
            else:
                assert got == _exact_dequant(c, s, g), (hex(s), c)


def test_double_rounding_cases_exist_and_are_single_rounded():
    """Find (code, scale, g) triples where rounding to float32 first would change the
    BF16 result, and check that the oracle rounds them once."""
    found = 0
    r = np.random.default_rng(3)
    for d in r.uniform(1.0, 5000.0, size=400).astype(np.float32):
        g = formats.global_multiplier(d, True)
        for c in (3, 5, 6, 7):
            for s in range(0x08, 0x7F):
                exact = e2m1_exact(c) * e4m3_exact(s) * f32_exact(g)
                once = bf16_round_exact(exact)
                twice = bf16_round_exact(Fraction(float(np.float32(float(exact)))))
                if once != twice:
                    codes = np.zeros((1, 16), dtype=np.uint8)
                    codes[0, 0] = c
                    w = dense.dequant(_pack(codes), np.array([[s]], dtype=np.uint8), d, True, 16)
                    assert int(w[0, 0]) == once
                    found += 1
    assert found > 0


def test_gemm_brute_force_4x16x16():
    c = synth.uniform_codes_case(M=4, K=16, N=16, seed=99)
    y, yb = dense.linear(c.x_bits, c.packed, c.scales, c.divisor, True)
    g = formats.global_multiplier(c.divisor, True)
    codes = dense.unpack_codes(c.packed, 16)
    for m in range(4):
        for n in range(16):
            acc = Fraction(0)
            for k in range(16):
                wb = _exact_dequant(int(codes[n, k]), int(c.scales[n, k // 16]), g)
                acc += bf16_exact(int(c.x_bits[m, k])) * bf16_exact(wb)
            assert abs(Fraction(float(y[m, n])) - acc) <= abs(acc) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 140)
            assert int(yb[m, n]) == bf16_round_exact(acc)


def test_gemm_power_of_two_scales_is_exact():
    """With power-of-two scales and global, every weight is the exact code value times
    a power of two, so Y is the exact dot product rounded once."""
    r = synth.rng(5)
    M, K, N = 3, 64, 8
    codes = r.integers(0, 16, size=(N, K), dtype=np.uint8)
    scales = r.choice(np.array([0x30, 0x38, 0x40, 0x48, 0x20], dtype=np.uint8), size=(N, K // 16))
    x = synth.normal_bf16(r, (M, K))
    y, yb = dense.linear(x, _pack(codes), scales, 0.25, False)
    for m in range(M):
        for n in range(N):
            acc = sum(bf16_exact(int(x[m, k])) * e2m1_exact(int(codes[n, k]))
                      * e4m3_exact(int(scales[n, k // 16])) * Fraction(1, 4) for k in range(K))
            assert Fraction(float(y[m, n])) == acc or abs(Fraction(float(y[m, n])) - acc) < abs(acc) * Fraction(1, 2 ** 50)
            assert int(yb[m, n]) == bf16_round_exact(acc)


def test_dequant_quant_idempotent():
    r = synth.rng(21)
    w = synth.normal_weight(r, 64, 256)
    p1, s1, d = synth.quantize(w)
    w1 = dense.dequant(p1, s1, d, True, 256)
    p2, s2, _ = synth.quantize(formats.bf16_to_float(w1).astype(np.float32), divisor=d)
    w2 = dense.dequant(p2, s2, d, True, 256)
    assert np.array_equal(w1, w2)
    assert np.array_equal(p1, p2) and np.array_equal(s1, s2)


def test_quantized_weight_is_close_to_source():
    r = synth.rng(22)
    w = synth.normal_weight(r, 128, 512)
    p, s, d = synth.quantize(w)
    assert abs(float(np.abs(w).max()) * float(d) - 2688.0) < 1e-2
    wd = formats.bf16_to_float(dense.dequant(p, s, d, True, 512))
    err = np.linalg.norm(wd - w) / np.linalg.norm(w)
    assert 0.03 < err < 0.15          # 4-bit E2M1 with 16-element groups


def test_awq_identity_and_dropped_scale_control():
    c = synth.gaussian_case(8, 256, 64, seed=31, awq=True)
    ones = np.full(c.K, 0x3F80, dtype=np.uint16)
    y0, _ = dense.linear(c.x_bits, c.packed, c.scales, c.divisor, True)
    y1, _ = dense.linear(c.x_bits, c.packed, c.scales, c.divisor, True, pqs_bits=ones)
    assert np.array_equal(y0, y1)
    ya, _ = dense.linear(c.x_bits, c.packed, c.scales, c.divisor, True, pqs_bits=c.pqs_bits)
    # dropping the scale must fail the parity tolerance by a wide margin
    rel = np.linalg.norm(y0 - ya) / np.linalg.norm(ya)
    assert rel > 0.2
    # the scaled activation is a single BF16 rounding of the exact product
    xs = dense.awq_scale_activation(c.x_bits[:2, :32], c.pqs_bits[:32])
    for m in range(2):
        for k in range(32):
            want = bf16_round_exact(bf16_exact(int(c.x_bits[m, k])) * bf16_exact(int(c.pqs_bits[k])))
            assert int(xs[m, k]) == want


def test_linear_row_sampling_matches_full():
    c = synth.gaussian_case(4, 128, 96, seed=41)
    y, yb = dense.linear(c.x_bits, c.packed, c.scales, c.divisor, True)
    rows = np.array([0, 5, 95, 17])
    ys, ysb = dense.linear(c.x_bits, c.packed, c.scales, c.divisor, True, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(ysb, yb[:, rows])


# ------------------------------------------------- FP16 activations ---
@pytest.mark.parametrize("divisor", [448.0, 3.0, 24366.764, 0.37, 1.0e-3, 1.0e6])
def test_dequant_f16_exact_over_all_codes_and_scales(divisor):
    """FP16 dequant of every (code, scale) pair against exact rational rounding,
    including products that overflow FP16 (1e-3) or fall in its subnormals (1e6)."""
    codes = np.tile(np.arange(16, dtype=np.uint8), (256, 1))
    scales = np.arange(256, dtype=np.uint8).reshape(256, 1)
    w = dense.dequant(_pack(codes), scales, divisor, True, 16, act="f16")
    g = formats.global_multiplier(divisor, True)
    for s in range(256):
        for c in range(16):
            got = int(w[s, c])
            if e4m3_exact(s) is None:
                assert got & 0x7FFF == 0x7E00
                assert (got >> 15) == (((c >> 3) ^ (s >> 7)) & 1)
            else:
                assert got == _exact_dequant(c, s, g, "f16"), (hex(s), c)


def test_f16_dequant_is_not_the_bf16_one():
    """Control: the two activation types give different weights for a generic global."""
    codes = np.tile(np.arange(16, dtype=np.uint8), (64, 1))
    scales = np.arange(0x20, 0x60, dtype=np.uint8).reshape(64, 1)
    wb = formats.bf16_to_float(dense.dequant(_pack(codes), scales, 24366.764, True, 16))
    wh = formats.f16_to_float(dense.dequant(_pack(codes), scales, 24366.764, True, 16, act="f16"))
    assert not np.array_equal(wb, wh)


def test_gemm_f16_brute_force_4x16x16():
    c = synth.uniform_codes_case(M=4, K=16, N=16, seed=98)
    x = synth.normal_act(synth.rng(5), (4, 16), "f16")
    y, yb = dense.linear(x, c.packed, c.scales, c.divisor, True, act="f16")
    g = formats.global_multiplier(c.divisor, True)
    codes = dense.unpack_codes(c.packed, 16)
    for m in range(4):
        for n in range(16):
            acc = Fraction(0)
            for k in range(16):
                wb = _exact_dequant(int(codes[n, k]), int(c.scales[n, k // 16]), g, "f16")
                acc += f16_exact(int(x[m, k])) * f16_exact(wb)
            assert abs(Fraction(float(y[m, n])) - acc) <= abs(acc) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 140)
            assert int(yb[m, n]) == f16_round_exact(acc)


def test_awq_f16_single_rounding_and_dropped_scale_control():
    c = synth.gaussian_case(8, 256, 64, seed=33, awq=True, act="f16")
    xs = dense.awq_scale_activation(c.x_bits[:2, :32], c.pqs_bits[:32], act="f16")
    for m in range(2):
        for k in range(32):
            want = f16_round_exact(f16_exact(int(c.x_bits[m, k])) * f16_exact(int(c.pqs_bits[k])))
            assert int(xs[m, k]) == want
    y0, _ = dense.linear(c.x_bits, c.packed, c.scales, c.divisor, True, act="f16")
    ya, _ = dense.linear(c.x_bits, c.packed, c.scales, c.divisor, True, pqs_bits=c.pqs_bits, act="f16")
    assert np.linalg.norm(y0 - ya) / np.linalg.norm(ya) > 0.2
