"""Helpers shared by the GPU parity tests: move synthetic cases to the device,
run the library through its C ABI binding, and compare with the oracle."""

import numpy as np
import torch

import w4a16_nvfp4_weight_gb300 as nv
from oracle import dense, formats

# Parity bar for floating-point outputs (GEMM / MoE), against the oracle's
# BF16-rounded output: relative Frobenius error and max-abs error relative to
# max|ref|.
REL_FRO = 2e-3
MAX_ABS = 2e-2


def bits_to_bf16_tensor(bits, device="cuda"):
    return bits_to_tensor(bits, "bf16", device)


def bits_to_tensor(bits, act, device="cuda"):
    """16-bit patterns -> a CUDA tensor of the activation type ("bf16" or "f16")."""
    a = np.ascontiguousarray(bits, dtype=np.uint16)
    dt = torch.bfloat16 if act == "bf16" else torch.float16
    return torch.from_numpy(a.view(np.int16)).view(dt).to(device)


def tensor_to_bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(device)


def repack_case(case, device="cuda"):
    return nv.repack(u8(case.packed, device), u8(case.scales, device), float(case.divisor),
                     case.N, case.K, global_is_divisor=True)


def compare(y_gpu_bits, y_ref_bits, what="", act="bf16"):
    """Assert the parity bar; returns (rel_fro, max_abs_rel)."""
    g = formats.act_to_float(y_gpu_bits, act)
    r = formats.act_to_float(y_ref_bits, act)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    assert np.all(np.isfinite(r)), f"{what}: non-finite oracle output"
    denom = np.linalg.norm(r)
    rel = np.linalg.norm(g - r) / denom if denom > 0 else np.linalg.norm(g - r)
    mx = np.abs(r).max() if r.size else 0.0
    mabs = np.abs(g - r).max() / mx if mx > 0 else np.abs(g - r).max() if g.size else 0.0
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel:.3e} > {REL_FRO}"
    assert mabs <= MAX_ABS, f"{what}: max-abs error {mabs:.3e} * max|ref| > {MAX_ABS}"
    return rel, mabs


def check_device_status():
    st = nv.device_status(clear=True)
    assert st == 0, f"device status word {st}"


def oracle_linear(case, rows=None, awq=True, act="bf16"):
    pqs = case.pqs_bits if awq else None
    return dense.linear(case.x_bits, case.packed, case.scales, case.divisor, True,
                        pqs_bits=pqs, rows=rows, act=act)
