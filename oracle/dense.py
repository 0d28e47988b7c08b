"""Dense W4A16 NVFP4 linear, the plain way (test infrastructure).

What the method computes ("[TRTLLM-12288][feat] Support Nemotron-H nvfp4 ckpt
on Hopper", Description and Changes table, linear row): dequantize the NVFP4
weight to BF16 every forward step, then run an ordinary BF16 GEMM
(cublas_mm / F.linear) on it.  The fused GPU kernels must reach exactly that
result up to FP32 summation order, so the oracle is that definition written
out:

1. W[n, k] = RN_bf16( e2m1(code[n, k]) * e4m3(scale[n, k // 16]) * g )
   -- the product is exact in float64 (2 + 4 + 24 significant bits) and is
   rounded once, to BF16, ties to even.  g is the FP32 global multiplier
   (the divisor form inverted first).
2. optional AWQ: x'[m, k] = RN_bf16( x[m, k] * pre_quant_scale[k] ) -- the
   stored weights are W/s, so the activation is multiplied by s before the
   GEMM, shape [1, hidden], and the product stays BF16 ("[None][fix] Apply the
   NVFP4_AWQ pre-quant scale in MegaMoE CuteDSL", Description and the commit
   that applies the scale on the CUTLASS W4A16 MoE path).
3. Y[m, n] = sum_k x'[m, k] * W[n, k] in float64 (every product of two BF16
   values is exact in float64); the reported output is RN_bf16(Y).

W4A16 covers FP16 activations as well as BF16 ("[TRTLLM-12720][feat] Support
nvfp4 w4a16 on sm120", Summary: "BF16/FP16 activations").  With ``act="f16"``
every BF16 rounding above is an FP16 rounding instead: the weight is
dequantized to the activation type (W = RN_f16 of the same exact product, so
one rounding still), x' = RN_f16(x * s), and the output is RN_f16(Y).

Packed layout of the inputs (the checkpoint form): ``packed`` uint8 [N, K/2],
row-major, the LOW nibble holding the even k; ``scales`` uint8 float8_e4m3fn
codes [N, K/16], row-major.  K must be a multiple of 16 (the group size).

Parity: pinned by tests/test_oracle_dense.py (worked codebook row, divisor
inversion worked values, exact rational rounding over all 16 x 256 code/scale
pairs, brute-force float64 dot products on 4x16x16, the power-of-two special
case, dequant(quant(x)) idempotence, AWQ identity and dropped-scale controls).
"""

import numpy as np

from .formats import act_bits, act_nan_bits, act_to_float, e2m1_value, e4m3_value, global_multiplier

GROUP = 16


def unpack_codes(packed, K):
    """uint8 [N, K/2] -> E2M1 codes int64 [N, K]; low nibble = even k."""
    p = np.asarray(packed, dtype=np.uint8)
    N = p.shape[0]
    codes = np.empty((N, K), dtype=np.int64)
    codes[:, 0::2] = p & 0xF
    codes[:, 1::2] = p >> 4
    return codes


def dequant_values(packed, scales, g, K):
    """Exact float64 products e2m1(code) * e4m3(scale) * g, shape [N, K]."""
    codes = unpack_codes(packed, K)
    s = e4m3_value(np.asarray(scales, dtype=np.uint8))           # [N, K/16]
    s_per_k = np.repeat(s, GROUP, axis=1)                         # [N, K]
    g64 = np.float64(np.float32(g))
    with np.errstate(invalid="ignore", over="ignore"):
        return e2m1_value(codes) * s_per_k * g64


def dequant(packed, scales, global_scale, global_is_divisor, K, act="bf16"):
    """Bit patterns (uint16 [N, K]) of the weight dequantized to ``act``."""
    g = global_multiplier(global_scale, global_is_divisor)
    v = dequant_values(packed, scales, g, K)
    bits = act_bits(v, act)
    # A NaN weight (only from a NaN scale code) carries the sign of the product
    # of the code's and the scale's signs, like the finite weights do.
    nan = np.isnan(v)
    if nan.any():
        codes = unpack_codes(packed, K)
        sc = np.repeat(np.asarray(scales, dtype=np.uint8).astype(np.int64), GROUP, axis=1)
        sgn = ((codes >> 3) ^ (sc >> 7) ^ int(np.signbit(g))) & 1
        bits = np.where(nan, (act_nan_bits(act) | (sgn << 15)).astype(np.uint16), bits)
    return bits


def awq_scale_activation(x_bits, pqs_bits, act="bf16"):
    """x' = RN(x * pre_quant_scale) in the activation type, broadcast over rows
    (uint16 in/out)."""
    x = act_to_float(x_bits, act)
    s = act_to_float(np.asarray(pqs_bits).reshape(1, -1), act)
    return act_bits(x * s, act)


def gemm(x_bits, w_bits, act="bf16"):
    """Y = X . W^T in float64 from 16-bit operands X [M, K], W [N, K]."""
    x = act_to_float(x_bits, act)
    w = act_to_float(w_bits, act)
    return x @ w.T


def linear(x_bits, packed, scales, global_scale, global_is_divisor, pqs_bits=None, rows=None, act="bf16"):
    """Full W4A16 linear.  Returns (Y_float64 [M, N'], Y_bits [M, N']) with the
    output rounded to the activation type ``act`` ("bf16" or "f16").

    ``rows`` optionally restricts the output to a subset of the N output
    features (the oracle then dequantizes only those weight rows), for
    sampled checks at sizes where the whole matrix is too slow.
    """
    K = np.asarray(x_bits).shape[1]
    p = np.asarray(packed)
    s = np.asarray(scales)
    if rows is not None:
        p = p[rows]
        s = s[rows]
    w = dequant(p, s, global_scale, global_is_divisor, K, act)
    x = x_bits if pqs_bits is None else awq_scale_activation(x_bits, pqs_bits, act)
    y = gemm(x, w, act)
    return y, act_bits(y, act)
