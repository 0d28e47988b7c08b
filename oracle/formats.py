"""Number formats of NVFP4 weights, decoded the plain way (test infrastructure).

* E2M1 (FP4) element codes -- "E2M1 FP4 codebook lookup" ("[TRTLLM-12288][feat]
  Support Nemotron-H nvfp4 ckpt on Hopper", Changes table, Triton NVFP4
  dequantization row).  A 4-bit code is a sign bit (bit 3) and a 3-bit index
  into the magnitude codebook {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* E4M3 group scales -- "E4M3 group scales" with group size 16 (SGLang PR 40022,
  Motivation); the FP8 type is float8_e4m3fn (the FN variant: no infinities,
  one NaN pattern per sign, maximum 448).
* the FP32 per-tensor global scale, which compressed-tensors checkpoints store
  as a divisor (1/scale) and which must be inverted before use (SGLang PR
  40022, "Note the global-scale inversion").
* BF16 round-to-nearest-even of an exact float64 value, and the same for
  FP16 (IEEE binary16), the other 16-bit activation type of W4A16 ("BF16/FP16
  activations": "[TRTLLM-12720][feat] Support nvfp4 w4a16 on sm120", Summary).

Parity: pinned by tests/test_oracle_formats.py (hand-listed codebook row,
closed-form E2M1 from its exponent/mantissa fields, all 256 E4M3 codes against
torch.float8_e4m3fn, BF16 and FP16 rounding against torch's float32 casts and
against exact rational rounding).
"""

import numpy as np

# Magnitudes of the eight unsigned E2M1 codes (code & 7), as printed by the
# format's codebook.
E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e2m1_value(codes):
    """Decode E2M1 codes (integers 0..15) to float64.

    Bit 3 is the sign; bits 0..2 index the codebook.  Code 0x8 decodes to -0.0.
    """
    c = np.asarray(codes).astype(np.int64)
    mag = np.asarray(E2M1_MAGNITUDES, dtype=np.float64)[c & 7]
    return np.where((c & 8) != 0, -mag, mag)


def e4m3_value(codes):
    """Decode float8_e4m3fn codes (integers 0..255) to float64 by the closed form.

    sign = bit 7, exponent = bits 3..6 (bias 7), mantissa = bits 0..2.
    exponent 0        -> subnormal  m/8 * 2**-6
    exponent 15, m 7  -> NaN (the FN variant has no infinities)
    otherwise         -> (1 + m/8) * 2**(e - 7)
    """
    c = np.asarray(codes).astype(np.int64)
    sign = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 7
    sub = m.astype(np.float64) / 8.0 * 2.0 ** -6
    norm = (1.0 + m.astype(np.float64) / 8.0) * np.exp2((e - 7).astype(np.float64))
    mag = np.where(e == 0, sub, norm)
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def global_multiplier(stored, stored_is_divisor):
    """The FP32 multiplier g applied to every weight of a tensor.

    A checkpoint that stores the global scale as a divisor d gets
    g = RN_fp32(1/d) -- one IEEE float32 division -- before any weight is
    formed (SGLang PR 40022, "Note the global-scale inversion": without it the
    BF16 dequant overflows).  Otherwise g is the stored float32 value.
    """
    s = np.float32(stored)
    if stored_is_divisor:
        with np.errstate(divide="ignore"):
            return np.float32(np.float32(1.0) / s)
    return s


_BF16_MIN_NORMAL = 2.0 ** -126


def bf16_bits(values):
    """Round exact float64 values to BF16 (round to nearest, ties to even).

    Returns the 16-bit patterns as uint16.  BF16 has 8 significant bits, the
    float32 exponent range and subnormals down to 2**-133.  Values whose
    rounded magnitude reaches 2**128 become infinity.  NaN becomes the quiet
    pattern 0x7FC0 with the value's sign bit; -0.0 keeps its sign.

    The rounding is done once, on the float64 value, by scaling the magnitude
    so that one unit in the last BF16 place is 1.0, rounding to an integer with
    numpy's rint (ties to even) and scaling back; all three steps are exact in
    float64 for the magnitudes involved.
    """
    v = np.asarray(values, dtype=np.float64)
    sign = np.signbit(v).astype(np.uint32) << 15
    a = np.abs(v)
    finite = np.isfinite(a)
    a_f = np.where(finite, a, 0.0)
    _, e = np.frexp(a_f)                       # a = m * 2**e, m in [0.5, 1)
    quantum_exp = np.where(a_f >= _BF16_MIN_NORMAL, e - 8, -133)
    r = np.rint(np.ldexp(a_f, -quantum_exp))  # integer significand, RNE
    rounded = np.ldexp(r, quantum_exp)        # exact float64, BF16-representable
    overflow = rounded >= 2.0 ** 128
    with np.errstate(over="ignore"):
        f32 = np.where(overflow, 0.0, rounded).astype(np.float32)
    bits = (f32.view(np.uint32) >> 16).astype(np.uint32)
    bits = np.where(overflow | np.isinf(a), 0x7F80, bits)
    bits = np.where(np.isnan(a), 0x7FC0, bits)
    return (bits | sign).astype(np.uint16)


def bf16_to_float(bits):
    """Exact float64 value of BF16 bit patterns (uint16)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


_F16_MIN_NORMAL = 2.0 ** -14


def f16_bits(values):
    """Round exact float64 values to FP16 (IEEE binary16; nearest, ties to even).

    Returns the 16-bit patterns as uint16.  FP16 has 11 significant bits,
    exponent bias 15 and subnormals down to 2**-24; values whose rounded
    magnitude reaches 2**16 become infinity (the largest finite value is
    65504).  NaN becomes the quiet pattern 0x7E00 with the value's sign bit;
    -0.0 keeps its sign.  One rounding of the float64 value, done as for BF16:
    scale so that one unit in the last FP16 place is 1.0, rint, scale back.
    """
    v = np.asarray(values, dtype=np.float64)
    sign = np.signbit(v).astype(np.uint32) << 15
    a = np.abs(v)
    finite = np.isfinite(a)
    a_f = np.where(finite, a, 0.0)
    _, e = np.frexp(a_f)                       # a = m * 2**e, m in [0.5, 1)
    quantum_exp = np.where(a_f >= _F16_MIN_NORMAL, e - 11, -24)
    r = np.rint(np.ldexp(a_f, -quantum_exp))  # integer significand, RNE
    rounded = np.ldexp(r, quantum_exp)        # exact float64, FP16-representable
    overflow = rounded >= 2.0 ** 16
    h = np.where(overflow, 0.0, rounded).astype(np.float16)   # exact: representable
    bits = h.view(np.uint16).astype(np.uint32)
    bits = np.where(overflow | np.isinf(a), 0x7C00, bits)
    bits = np.where(np.isnan(a), 0x7E00, bits)
    return (bits | sign).astype(np.uint16)


def f16_to_float(bits):
    """Exact float64 value of FP16 bit patterns (uint16)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


ACTIVATION_TYPES = ("bf16", "f16")


def act_bits(values, act):
    """Round to the activation type: ``act`` is "bf16" or "f16"."""
    if act == "bf16":
        return bf16_bits(values)
    if act == "f16":
        return f16_bits(values)
    raise ValueError(f"unknown activation type {act!r}")


def act_to_float(bits, act):
    if act == "bf16":
        return bf16_to_float(bits)
    if act == "f16":
        return f16_to_float(bits)
    raise ValueError(f"unknown activation type {act!r}")


def act_nan_bits(act):
    """The quiet-NaN pattern (sign bit clear) the rounding functions produce."""
    return 0x7FC0 if act == "bf16" else 0x7E00


def swizzled_scale_offset(n, j, G):
    """Byte offset of the scale of row n, 16-group j in the swizzled checkpoint
    layout of a weight with G = K/16 groups per row.

    The pages keep NVFP4 per-block scales in a swizzled layout and derive the
    linear [N, K/16] view from it ("[TRTLLM-12288][feat] Support Nemotron-H
    nvfp4 ckpt on Hopper", Linear section: "Per-block scales stay in swizzled
    layout; the unswizzled view is a derived non-persistent buffer"), without
    printing the layout.  The reading taken: the 128 x 4 tiles of NVIDIA's
    block-scaled GEMMs -- rows padded to 128 and groups to 4, tiles of 128 rows
    x 4 groups stored row-tile-major as 512 bytes each, and inside a tile the
    scale of (r, c) at (r % 32) * 16 + (r // 32) * 4 + c.
    """
    n = np.asarray(n, dtype=np.int64)
    j = np.asarray(j, dtype=np.int64)
    tiles_per_row = (int(G) + 3) // 4
    tile = (n // 128) * tiles_per_row + j // 4
    r, c = n % 128, j % 4
    return tile * 512 + (r % 32) * 16 + (r // 32) * 4 + c


def swizzled_scales_size(N, K):
    """Bytes of the swizzled scale tensor of an N x K weight."""
    G = K // 16
    return ((N + 127) // 128 * 128) * ((G + 3) // 4 * 4)


def unswizzle_scales(swizzled, N, K):
    """Linear scale codes uint8 [N, K/16] from the swizzled bytes."""
    G = K // 16
    sw = np.asarray(swizzled, dtype=np.uint8).reshape(-1)
    n = np.arange(N)[:, None]
    j = np.arange(G)[None, :]
    return sw[swizzled_scale_offset(n, j, G)]
