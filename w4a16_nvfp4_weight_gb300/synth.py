"""Seeded synthetic inputs shaped like the dense, LM-head and MoE workloads.

This module only *makes inputs*: random numbers, the BF16 or FP16 cast of
activations (torch's float32->bfloat16 / float16 casts) and the weight quantizer that turns an
FP32 matrix into NVFP4 checkpoint tensors (packed E2M1 codes, E4M3 group
scales, an FP32 global divisor).  It contains no decoding, dequantization,
GEMM or routing arithmetic; both the CUDA library's tests and the CPU oracle
consume what it produces, and neither is imported here.

Quantizer (the input recipe of the workloads; the checkpoint stores the global
scale as a divisor d, which the kernel side inverts -- SGLang PR 40022, "Note
the global-scale inversion"):

* d = 448 * 6 / absmax(W)                                (float32)
* s[n, g] = E4M3_satfinite_RNE( absmax(W[n, 16g:16g+16]) / 6 * d )
* code[n, k] = E2M1_RNE( W[n, k] * d / s[n, k // 16] ), saturated at +-6;
  a group whose scale is 0 gets code 0 everywhere.
* E2M1 rounding is to the nearest codebook magnitude, ties to the code with an
  even mantissa bit (0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4).
* packed[n, k // 2] holds code[n, k] in the low nibble for even k.

Seeds: a workload's seed is ``1234 + 1000 * workload_index + shape_index``.
"""

import numpy as np
import torch

E4M3_MAX = 448.0
E2M1_MAX = 6.0


def rng(seed):
    return np.random.Generator(np.random.PCG64(int(seed)))


def seed_for(workload_index, shape_index):
    return 1234 + 1000 * int(workload_index) + int(shape_index)


def bf16_bits_of(x_f32):
    """BF16 bit patterns (uint16) of float32 values, via torch's RNE cast."""
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def f16_bits_of(x_f32):
    """FP16 bit patterns (uint16) of float32 values, via torch's RNE cast."""
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32))
    return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16).copy()


def act_bits_of(x_f32, act):
    """16-bit activation patterns: act = "bf16" or "f16"."""
    return bf16_bits_of(x_f32) if act == "bf16" else f16_bits_of(x_f32)


def normal_bf16(r, shape, std=1.0):
    return normal_act(r, shape, "bf16", std)


def normal_act(r, shape, act, std=1.0):
    x = r.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x = x * np.float32(std)
    return act_bits_of(x, act)


def _e4m3_codes(v_f32):
    """float32 -> float8_e4m3fn codes (uint8), saturating to +-448, RNE (torch cast)."""
    v = np.clip(np.asarray(v_f32, dtype=np.float32), -E4M3_MAX, E4M3_MAX)
    t = torch.from_numpy(np.ascontiguousarray(v)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def _e4m3_float(codes_u8):
    t = torch.from_numpy(np.ascontiguousarray(codes_u8, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float32).numpy()


# Rounding thresholds of |v| onto codebook index 0..7, with the tie direction
# that keeps the mantissa bit even: (threshold, tie_goes_up).
_E2M1_STEPS = ((0.25, False), (0.75, True), (1.25, False), (1.75, True),
               (2.5, False), (3.5, True), (5.0, False))


def _e2m1_codes(v):
    a = np.abs(v)
    idx = np.zeros(v.shape, dtype=np.uint8)
    for thr, up in _E2M1_STEPS:
        idx += (a >= thr) if up else (a > thr)
    sign = (v < 0) & (idx > 0)
    return (idx | (sign.astype(np.uint8) << 3)).astype(np.uint8)


def quantize(w, divisor=None, row_chunk=4096):
    """FP32 weight [N, K] -> (packed uint8 [N, K/2], scales uint8 [N, K/16], d float32)."""
    w = np.asarray(w, dtype=np.float32)
    N, K = w.shape
    assert K % 16 == 0, "K must be a multiple of the group size 16"
    if divisor is None:
        amax = float(np.abs(w).max())
        divisor = np.float32(E4M3_MAX * E2M1_MAX) / np.float32(amax if amax > 0 else 1.0)
    d = np.float32(divisor)
    packed = np.empty((N, K // 2), dtype=np.uint8)
    scales = np.empty((N, K // 16), dtype=np.uint8)
    for r0 in range(0, N, row_chunk):
        blk = w[r0:r0 + row_chunk].reshape(-1, K // 16, 16)
        gmax = np.abs(blk).max(axis=2)
        s_codes = _e4m3_codes(gmax / np.float32(E2M1_MAX) * d)
        s_val = _e4m3_float(s_codes).astype(np.float64)
        with np.errstate(divide="ignore", invalid="ignore"):
            v = blk.astype(np.float64) * np.float64(d) / s_val[:, :, None]
        v = np.where(s_val[:, :, None] > 0, v, 0.0)
        codes = _e2m1_codes(v).reshape(-1, K)
        packed[r0:r0 + row_chunk] = codes[:, 0::2] | (codes[:, 1::2] << 4)
        scales[r0:r0 + row_chunk] = s_codes
    return packed, scales, d


def normal_weight(r, N, K, std=0.02):
    return r.standard_normal(size=(N, K), dtype=np.float32) * np.float32(std)


class DenseCase:
    """One dense W4A16 linear problem (host numpy arrays)."""

    def __init__(self, M, K, N, x_bits, packed, scales, divisor, pqs_bits=None):
        self.M, self.K, self.N = M, K, N
        self.x_bits = x_bits          # uint16 [M, K]
        self.packed = packed          # uint8 [N, K/2]
        self.scales = scales          # uint8 [N, K/16]
        self.divisor = divisor        # float32 global scale stored as a divisor
        self.pqs_bits = pqs_bits      # uint16 [K] or None


def uniform_codes_case(M=4, K=256, N=256, seed=None):
    """The tiny linear: uniform random 4-bit codes, scales uniform over the
    positive finite E4M3 codes in [2**-4, 448] (0x18..0x7E), divisor 448."""
    r = rng(seed_for(0, 0) if seed is None else seed)
    codes = r.integers(0, 16, size=(N, K), dtype=np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    scales = r.integers(0x18, 0x7F, size=(N, K // 16), dtype=np.uint8)
    x = normal_bf16(r, (M, K))
    return DenseCase(M, K, N, x, packed, scales, np.float32(448.0))


def awq_scale_bits(r, K, act="bf16"):
    """Per-channel AWQ pre-quant scale, log-uniform in [1/e, e], as BF16 (or FP16)."""
    return act_bits_of(np.exp(r.uniform(-1.0, 1.0, size=K)).astype(np.float32), act)


def gaussian_case(M, K, N, seed, awq=False, act="bf16"):
    """A linear whose weight is quantized from N(0, 0.02); X ~ N(0, 1) in the
    activation type ``act`` ("bf16" or "f16")."""
    r = rng(seed)
    w = normal_weight(r, N, K)
    packed, scales, d = quantize(w)
    del w
    x = normal_act(r, (M, K), act)
    pqs = awq_scale_bits(r, K, act) if awq else None
    return DenseCase(M, K, N, x, packed, scales, d, pqs)


def weight_only(K, N, seed):
    """Quantized weight tensors of a gaussian linear, without activations."""
    r = rng(seed)
    w = normal_weight(r, N, K)
    return quantize(w)


class MoECase:
    def __init__(self, T, E, topk, H, I, x_bits, logits, fc1, fc2, pqs_bits=None):
        self.T, self.E, self.topk, self.H, self.I = T, E, topk, H, I
        self.x_bits = x_bits      # uint16 [T, H]
        self.logits = logits      # float32 [T, E]
        self.fc1 = fc1            # E x (packed [2I, H/2], scales [2I, H/16], divisor)
        self.fc2 = fc2            # E x (packed [H, I/2], scales [H, I/16], divisor)
        self.pqs_bits = pqs_bits  # uint16 [H] or None


def moe_weights(E, H, I, seed):
    r = rng(seed)
    fc1, fc2 = [], []
    for _ in range(E):
        fc1.append(quantize(normal_weight(r, 2 * I, H)))
        fc2.append(quantize(normal_weight(r, H, I)))
    return fc1, fc2


def moe_case(T, seed, E=128, topk=8, H=2048, I=768, weights=None, awq=False, act="bf16"):
    """MoE layer inputs: logits ~ N(0,1) FP32, X ~ N(0,1) BF16 (or FP16), experts
    from N(0,0.02)."""
    fc1, fc2 = weights if weights is not None else moe_weights(E, H, I, seed + 500)
    r = rng(seed)
    logits = r.standard_normal(size=(T, E), dtype=np.float32)
    x = normal_act(r, (T, H), act)
    pqs = awq_scale_bits(r, H, act) if awq else None
    return MoECase(T, E, topk, H, I, x, logits, fc1, fc2, pqs)
