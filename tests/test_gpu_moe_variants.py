"""GPU parity of the MoE layer variants against the CPU oracle: non-gated
relu2 / silu experts, gate and up projections repacked as shards with their own
global scales, and the AWQ scale finalization max over experts of max(w3, w1).
Streaming (few rows per expert) and tile (many rows per expert) paths, BF16 and
FP16 activations."""

import numpy as np
import pytest
import torch

import w4a16_nvfp4_weight_gb300 as nv
from oracle import moe as omoe
from tests import gpu_util as gu
from w4a16_nvfp4_weight_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    torch.cuda.init()
    yield


def _stack(weights, N, K):
    """Repack the (packed, scales, divisor) tuples back to back."""
    size = nv.repack_size(N, K)
    buf = torch.empty(len(weights) * size, dtype=torch.uint8, device="cuda")
    for i, (p, s, d) in enumerate(weights):
        nv.repack(gu.u8(p), gu.u8(s), float(d), N, K, out=buf[i * size:(i + 1) * size])
    return buf


def _case(T, E, topk, H, I, seed, kind, act="bf16", awq=False):
    r = synth.rng(seed)
    fc1, fc2 = [], []
    for _ in range(E):
        if kind == "split":
            fc1.append((synth.quantize(synth.normal_weight(r, I, H)), synth.quantize(synth.normal_weight(r, I, H))))
        elif kind == "gated":
            fc1.append(synth.quantize(synth.normal_weight(r, 2 * I, H)))
        else:
            fc1.append(synth.quantize(synth.normal_weight(r, I, H)))
        fc2.append(synth.quantize(synth.normal_weight(r, H, I)))
    c = synth.moe_case(T, seed + 1, E=E, topk=topk, H=H, I=I, weights=(fc1, fc2), act=act, awq=awq)
    return c, fc1, fc2


def _run(c, fc1_dev, fc2_dev, act, activation, split, awq):
    x = gu.bits_to_tensor(c.x_bits, act)
    logits = torch.from_numpy(np.ascontiguousarray(c.logits)).cuda()
    pqs = gu.bits_to_tensor(c.pqs_bits, act) if awq else None
    out, routing = nv.moe_grouped(x, logits, fc1_dev, fc2_dev, c.topk, c.I, fc1_pre_quant_scale=pqs,
                                  return_routing=True, activation=activation, fc1_split=split)
    gu.check_device_status()
    return gu.tensor_to_bits(out), {k: v.cpu().numpy() for k, v in routing.items()}


# (5, 4, 2, 128, 128): streaming; (300, 4, 2, 256, 256): tile (150 rows per expert)
@pytest.mark.parametrize("T,E,topk,H,I", [(5, 4, 2, 128, 128), (300, 4, 2, 256, 256)])
@pytest.mark.parametrize("activation", ["relu2", "silu"])
@pytest.mark.parametrize("act", ["bf16", "f16"])
def test_non_gated_experts(T, E, topk, H, I, activation, act):
    c, fc1, fc2 = _case(T, E, topk, H, I, seed=T + I + len(activation), kind="plain", act=act, awq=(T == 300))
    out, routing = _run(c, _stack(fc1, I, H), _stack(fc2, H, I), act, activation, False, awq=(T == 300))
    ref = omoe.moe_layer(c.x_bits, c.logits, [(p, s, d, True) for p, s, d in fc1],
                         [(p, s, d, True) for p, s, d in fc2], topk, act=act, activation=activation,
                         pqs_bits=c.pqs_bits if T == 300 else None)
    assert np.array_equal(routing["perm"], ref["perm"])
    gu.compare(out, ref["out_bits"], f"{activation} T={T} {act}", act=act)


@pytest.mark.parametrize("T,E,topk,H,I", [(7, 4, 2, 128, 128), (64, 16, 4, 256, 128), (300, 4, 2, 256, 256)])
@pytest.mark.parametrize("act", ["bf16", "f16"])
def test_gate_up_shards_with_own_globals(T, E, topk, H, I, act):
    c, fc1, fc2 = _case(T, E, topk, H, I, seed=2 * T + I, kind="split", act=act)
    shards = [w for pair in fc1 for w in pair]                     # gate_0, up_0, gate_1, up_1, ...
    out, _ = _run(c, _stack(shards, I, H), _stack(fc2, H, I), act, "swiglu", True, awq=False)
    ref = omoe.moe_layer(c.x_bits, c.logits, [((gp, gs, gd, True), (up, us, ud, True)) for (gp, gs, gd), (up, us, ud) in fc1],
                         [(p, s, d, True) for p, s, d in fc2], topk, act=act, fc1_split=True)
    gu.compare(out, ref["out_bits"], f"shards T={T} {act}", act=act)


@pytest.mark.parametrize("T", [7, 300])
def test_shards_with_a_shared_global_match_the_fused_layer_bitwise(T):
    """One divisor for both halves: the shard layout must reproduce the fused
    [2I, H] layer bit for bit (same kernels, same sums, two tables)."""
    E, topk, H, I = 4, 2, 256, 256
    c, fc1, fc2 = _case(T, E, topk, H, I, seed=9 + T, kind="gated")
    shards = []
    for p, s, d in fc1:
        shards += [(p[:I], s[:I], d), (p[I:], s[I:], d)]
    fused, _ = _run(c, _stack(fc1, 2 * I, H), _stack(fc2, H, I), "bf16", "swiglu", False, awq=False)
    split, _ = _run(c, _stack(shards, I, H), _stack(fc2, H, I), "bf16", "swiglu", True, awq=False)
    assert np.array_equal(fused, split)


@pytest.mark.parametrize("act", ["bf16", "f16"])
def test_finalize_pre_quant_scale(act):
    r = synth.rng(71)
    E, H = 6, 2048
    w1 = np.stack([synth.awq_scale_bits(r, H, act) for _ in range(E)])
    w3 = np.stack([synth.awq_scale_bits(r, H, act) for _ in range(E)])
    got = nv.moe_finalize_pre_quant_scale(gu.bits_to_tensor(w1, act), gu.bits_to_tensor(w3, act))
    assert np.array_equal(gu.tensor_to_bits(got), omoe.finalize_pre_quant_scale(w1, w3, act))


def test_variant_arguments_rejected_on_host():
    x = torch.zeros((2, 64), dtype=torch.bfloat16, device="cuda")
    lg = torch.zeros((2, 2), dtype=torch.float32, device="cuda")
    w = torch.zeros(nv.repack_size(64, 64) * 4, dtype=torch.uint8, device="cuda")
    with pytest.raises(nv.Nvfp4Error):
        nv.moe_grouped(x, lg, w, w, 1, 64, activation="gelu")
    with pytest.raises(nv.Nvfp4Error):
        nv.moe_grouped(x, lg, w, w, 1, 64, activation="relu2", fc1_split=True)
