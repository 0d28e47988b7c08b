"""GPU parity of the persistent streaming MoE kernels against the CPU oracle.

With many (work item, column group) units the streaming path runs one wave of
CTAs that walk the units with K whole (moe_plan path "stream_persistent").
These cases are sized so that the plan takes that path on a GB300 (and on any
GPU with up to 256 SMs), at oracle sizes: gated SwiGLU experts with 8-, 16- and
32-row items, AWQ with its dropped-scale control, FP16 activations, non-gated
relu2 / silu experts, gate/up shards with their own globals, and run-to-run
bitwise determinism.  The bar is the GEMM parity bar against the oracle's
output; the routing tables are compared bit for bit.
"""

import numpy as np
import pytest
import torch

import w4a16_nvfp4_weight_gb300 as nv
from oracle import moe as omoe
from tests import gpu_util as gu
from w4a16_nvfp4_weight_gb300 import synth

pytestmark = pytest.mark.gpu


def _stack(weights, N, K):
    size = nv.repack_size(N, K)
    buf = torch.empty(len(weights) * size, dtype=torch.uint8, device="cuda")
    for i, (p, s, d) in enumerate(weights):
        nv.repack(gu.u8(p), gu.u8(s), float(d), N, K, out=buf[i * size:(i + 1) * size])
    return buf


def _case(T, E, topk, H, I, seed, kind="gated", act="bf16", awq=False):
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


def _run(c, fc1_dev, fc2_dev, act="bf16", activation="swiglu", split=False, awq=False):
    x = gu.bits_to_tensor(c.x_bits, act)
    logits = torch.from_numpy(np.ascontiguousarray(c.logits)).cuda()
    pqs = gu.bits_to_tensor(c.pqs_bits, act) if awq else None
    out, routing = nv.moe_grouped(x, logits, fc1_dev, fc2_dev, c.topk, c.I, fc1_pre_quant_scale=pqs,
                                  return_routing=True, activation=activation, fc1_split=split)
    gu.check_device_status()
    return gu.tensor_to_bits(out), {k: v.cpu().numpy() for k, v in routing.items()}


def _assert_persistent(T, E, topk, H, I, rows, activation="swiglu"):
    plan = nv.moe_plan(T, E, topk, H, I, activation)
    assert plan == {"path": "stream_persistent", "rows_per_item": rows}, plan


def _oracle_plain(c, fc1, fc2, act="bf16", activation="swiglu", awq=False):
    return omoe.moe_layer(c.x_bits, c.logits, [(p, s, d, True) for p, s, d in fc1],
                          [(p, s, d, True) for p, s, d in fc2], c.topk, act=act, activation=activation,
                          pqs_bits=c.pqs_bits if awq else None)


# routed rows per expert on average: 8 -> 8-row items, 10 -> 16-row items,
# 16 -> 32-row items
@pytest.mark.parametrize("T,E,topk,H,I,rows", [(64, 64, 8, 256, 1024, 8), (80, 64, 8, 128, 1024, 16),
                                               (128, 64, 8, 128, 1024, 32)])
def test_persistent_gated_full_compare(T, E, topk, H, I, rows):
    _assert_persistent(T, E, topk, H, I, rows)
    c, fc1, fc2 = _case(T, E, topk, H, I, seed=T + E + I)
    out, routing = _run(c, _stack(fc1, 2 * I, H), _stack(fc2, H, I))
    ref = _oracle_plain(c, fc1, fc2)
    assert np.array_equal(routing["idx"].reshape(T, topk), ref["idx"])
    assert np.array_equal(routing["perm"], ref["perm"])
    assert np.array_equal(routing["offsets"], ref["offsets"])
    gu.compare(out, ref["out_bits"], f"persistent MoE T={T}")


def test_persistent_awq_and_dropped_scale_control():
    T, E, topk, H, I = 64, 64, 8, 128, 1024
    _assert_persistent(T, E, topk, H, I, 8)
    c, fc1, fc2 = _case(T, E, topk, H, I, seed=41, awq=True)
    fc1_dev, fc2_dev = _stack(fc1, 2 * I, H), _stack(fc2, H, I)
    out, _ = _run(c, fc1_dev, fc2_dev, awq=True)
    ref = _oracle_plain(c, fc1, fc2, awq=True)
    gu.compare(out, ref["out_bits"], "persistent MoE AWQ")
    plain, _ = _run(c, fc1_dev, fc2_dev, awq=False)
    with pytest.raises(AssertionError):
        gu.compare(plain, ref["out_bits"], "persistent MoE dropped AWQ")


def test_persistent_f16_activations():
    T, E, topk, H, I = 128, 64, 8, 128, 1024
    _assert_persistent(T, E, topk, H, I, 32)
    c, fc1, fc2 = _case(T, E, topk, H, I, seed=43, act="f16", awq=True)
    out, _ = _run(c, _stack(fc1, 2 * I, H), _stack(fc2, H, I), act="f16", awq=True)
    ref = _oracle_plain(c, fc1, fc2, act="f16", awq=True)
    gu.compare(out, ref["out_bits"], "persistent MoE f16", act="f16")


@pytest.mark.parametrize("activation", ["relu2", "silu"])
def test_persistent_non_gated_experts(activation):
    T, E, topk, H, I = 128, 128, 8, 128, 1024
    _assert_persistent(T, E, topk, H, I, 8, activation)
    c, fc1, fc2 = _case(T, E, topk, H, I, seed=47 + len(activation), kind="plain")
    out, _ = _run(c, _stack(fc1, I, H), _stack(fc2, H, I), activation=activation)
    ref = _oracle_plain(c, fc1, fc2, activation=activation)
    gu.compare(out, ref["out_bits"], f"persistent MoE {activation}")


def test_persistent_gate_up_shards_with_own_globals():
    T, E, topk, H, I = 64, 64, 8, 128, 1024
    _assert_persistent(T, E, topk, H, I, 8)
    c, fc1, fc2 = _case(T, E, topk, H, I, seed=53, kind="split")
    shards = [w for pair in fc1 for w in pair]
    out, _ = _run(c, _stack(shards, I, H), _stack(fc2, H, I), split=True)
    ref = omoe.moe_layer(c.x_bits, c.logits,
                         [((gp, gs, gd, True), (up, us, ud, True)) for (gp, gs, gd), (up, us, ud) in fc1],
                         [(p, s, d, True) for p, s, d in fc2], topk, fc1_split=True)
    gu.compare(out, ref["out_bits"], "persistent MoE shards")


def test_persistent_deterministic():
    T, E, topk, H, I = 128, 64, 8, 128, 1024
    c, fc1, fc2 = _case(T, E, topk, H, I, seed=59)
    fc1_dev, fc2_dev = _stack(fc1, 2 * I, H), _stack(fc2, H, I)
    a, _ = _run(c, fc1_dev, fc2_dev)
    b, _ = _run(c, fc1_dev, fc2_dev)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("T,E,topk,H,I,path", [(1, 8, 2, 128, 256, "single_token"), (3, 8, 2, 128, 256, "stream_split"),
                                               (64, 64, 8, 128, 1024, "stream_persistent"),
                                               (300, 8, 2, 256, 256, "tile")])
def test_corrupt_expert_header_is_reported_not_trapped(T, E, topk, H, I, path):
    """An expert whose repacked header does not match (its magic overwritten)
    on each MoE path: the kernels skip that expert's work, record status 7 in
    the device status word and finish; the next call with intact weights
    matches the oracle again."""
    assert nv.moe_plan(T, E, topk, H, I)["path"] == path
    c, fc1, fc2 = _case(T, E, topk, H, I, seed=61 + T)
    fc1_dev, fc2_dev = _stack(fc1, 2 * I, H), _stack(fc2, H, I)
    size = nv.repack_size(2 * I, H)
    routed = int(np.argmax(np.bincount(omoe.route(c.logits, topk)[0].ravel(), minlength=E)))
    saved = fc1_dev[routed * size:routed * size + 4].clone()
    fc1_dev[routed * size:routed * size + 4] = 0
    x = gu.bits_to_tensor(c.x_bits, "bf16")
    logits = torch.from_numpy(np.ascontiguousarray(c.logits)).cuda()
    nv.moe_grouped(x, logits, fc1_dev, fc2_dev, topk, I)
    assert nv.device_status(clear=True) == 7
    fc1_dev[routed * size:routed * size + 4] = saved
    out, _ = _run(c, fc1_dev, fc2_dev)
    gu.compare(out, _oracle_plain(c, fc1, fc2)["out_bits"], f"after a corrupt header ({path})")


@pytest.mark.parametrize("E,topk,H,I,act,activation,awq", [(8, 2, 128, 256, "bf16", "swiglu", False),
                                                           (64, 8, 256, 512, "bf16", "swiglu", True),
                                                           (256, 8, 128, 128, "f16", "swiglu", True),
                                                           (16, 1, 192, 320, "bf16", "relu2", False),
                                                           (40, 5, 128, 192, "f16", "silu", False)])
def test_single_token_layer(E, topk, H, I, act, activation, awq):
    """One token (the moe_plan path "single_token"): two kernels, each routing
    the token itself -- FC1 writes h_j per routing slot, FC2 sums p_j * y_j in
    slot order inside a cluster of the slots.  Output against the oracle, the
    routing outputs bit for bit, AWQ with its dropped-scale control, FP16,
    non-gated experts, run-to-run bitwise equality."""
    assert nv.moe_plan(1, E, topk, H, I, activation)["path"] == "single_token"
    kind = "gated" if activation == "swiglu" else "plain"
    c, fc1, fc2 = _case(1, E, topk, H, I, seed=E + topk + H, kind=kind, act=act, awq=awq)
    fc1_dev = _stack(fc1, 2 * I if kind == "gated" else I, H)
    fc2_dev = _stack(fc2, H, I)
    out, routing = _run(c, fc1_dev, fc2_dev, act=act, activation=activation, awq=awq)
    ref = _oracle_plain(c, fc1, fc2, act=act, activation=activation, awq=awq)
    assert np.array_equal(routing["idx"].reshape(1, topk), ref["idx"])
    assert np.array_equal(routing["perm"], ref["perm"])
    assert np.array_equal(routing["offsets"], ref["offsets"])
    assert np.allclose(routing["p"].reshape(1, topk), ref["p"], rtol=2e-6, atol=1e-7)
    gu.compare(out, ref["out_bits"], f"single token E={E} k={topk} {act} {activation}", act=act)
    again, _ = _run(c, fc1_dev, fc2_dev, act=act, activation=activation, awq=awq)
    assert np.array_equal(out, again)
    if awq:
        plain, _ = _run(c, fc1_dev, fc2_dev, act=act, activation=activation, awq=False)
        with pytest.raises(AssertionError):
            gu.compare(plain, ref["out_bits"], "single token dropped AWQ", act=act)


def test_single_token_gate_up_shards():
    E, topk, H, I = 16, 4, 128, 256
    assert nv.moe_plan(1, E, topk, H, I)["path"] == "single_token"
    c, fc1, fc2 = _case(1, E, topk, H, I, seed=71, kind="split")
    shards = [w for pair in fc1 for w in pair]
    out, _ = _run(c, _stack(shards, I, H), _stack(fc2, H, I), split=True)
    ref = omoe.moe_layer(c.x_bits, c.logits,
                         [((gp, gs, gd, True), (up, us, ud, True)) for (gp, gs, gd), (up, us, ud) in fc1],
                         [(p, s, d, True) for p, s, d in fc2], topk, fc1_split=True)
    gu.compare(out, ref["out_bits"], "single token shards")
