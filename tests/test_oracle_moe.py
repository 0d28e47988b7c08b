"""Pins for oracle.moe: routing, permutation tables, the expert layer.

Independent checks: hand-built logits with a known top-k (ties included),
closed-form routing weights, permutation invariants, the E=1 / top-1 case that
reduces to two dense linears, SiLU against scipy's logistic function, and a
pure-Python loop implementation of a tiny layer built on exact rational
dequantization (tests/exact.py).
"""

import math

import numpy as np
import pytest
from scipy.special import expit

from oracle import dense, formats, moe
from tests.exact import bf16_exact, bf16_round_exact, e2m1_exact, e4m3_exact, f16_exact, f16_round_exact, f32_exact
from w4a16_nvfp4_weight_gb300 import synth


def test_route_hand_built():
    E = 16
    l = np.zeros((3, E), dtype=np.float32)
    l[0] = np.arange(E, dtype=np.float32)                  # strictly increasing
    l[1, [3, 9, 12]] = 5.0                                  # three-way tie at the top
    l[1, 7] = 4.0
    l[2, :] = -1.0
    l[2, 15] = 2.0
    idx, p = moe.route(l, 4)
    assert idx[0].tolist() == [15, 14, 13, 12]
    assert idx[1].tolist() == [3, 9, 12, 7]                 # ties -> lower index first
    assert idx[2].tolist() == [15, 0, 1, 2]
    e = math.exp
    z0 = e(0) + e(-1) + e(-2) + e(-3)
    assert np.allclose(p[0], [1 / z0, e(-1) / z0, e(-2) / z0, e(-3) / z0], rtol=1e-15)
    z1 = 3 + e(-1)
    assert np.allclose(p[1], [1 / z1, 1 / z1, 1 / z1, e(-1) / z1], rtol=1e-15)
    for row in p:
        assert abs(row.sum() - 1.0) <= 2 ** -52 * 4


def test_route_negative_zero_ties_with_zero():
    l = np.array([[-0.0, 0.0, -1.0, 0.0]], dtype=np.float32)
    idx, _ = moe.route(l, 3)
    assert idx[0].tolist() == [0, 1, 3]


def test_permutation_invariants():
    r = np.random.default_rng(0)
    T, E, k = 37, 16, 4
    idx, _ = moe.route(r.standard_normal((T, E)).astype(np.float32), k)
    counts, offsets, perm, inv = moe.permute(idx, E)
    assert offsets[0] == 0 and offsets[-1] == T * k
    assert np.all(np.diff(offsets) == counts) and np.all(counts >= 0)
    assert sorted(perm.tolist()) == list(range(T * k))
    assert np.array_equal(inv[perm], np.arange(T * k))
    flat = idx.ravel()
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)                     # stable: token, then slot
    # empty routing
    c0, o0, p0, i0 = moe.permute(np.zeros((0, k), dtype=np.int32), E)
    assert o0.tolist() == [0] * (E + 1) and p0.size == 0


def test_silu_against_logistic():
    v = np.array([0.0, 1.0, -1.0, 20.0, -20.0, 3.5, -7.25])
    assert np.allclose(moe.silu(v), v * expit(v), rtol=1e-15, atol=0)
    assert moe.silu(0.0) == 0.0


def _tiny_layer(T=3, E=4, topk=2, H=32, I=16, seed=5, awq=False, act="bf16"):
    r = synth.rng(seed)
    fc1, fc2 = [], []
    for _ in range(E):
        fc1.append(synth.quantize(synth.normal_weight(r, 2 * I, H)))
        fc2.append(synth.quantize(synth.normal_weight(r, H, I)))
    return synth.moe_case(T, seed, E=E, topk=topk, H=H, I=I, weights=(fc1, fc2), awq=awq, act=act)


_ROUND = {"bf16": bf16_round_exact, "f16": f16_round_exact}
_VALUE = {"bf16": bf16_exact, "f16": f16_exact}


def _loop_dequant(packed, scales, divisor, K, act="bf16"):
    g = f32_exact(np.float32(1.0) / np.float32(divisor))
    N = packed.shape[0]
    out = []
    for n in range(N):
        row = []
        for k in range(K):
            byte = int(packed[n, k // 2])
            code = (byte & 0xF) if k % 2 == 0 else (byte >> 4)
            v = e2m1_exact(code) * e4m3_exact(int(scales[n, k // 16])) * g
            row.append(float(_VALUE[act](_ROUND[act](v))))
        out.append(row)
    return out


@pytest.mark.parametrize("act", ["bf16", "f16"])
def test_tiny_layer_against_python_loops(act):
    c = _tiny_layer(act=act)
    res = moe.moe_layer(c.x_bits, c.logits, [(p, s, d, True) for p, s, d in c.fc1],
                        [(p, s, d, True) for p, s, d in c.fc2], c.topk, act=act)
    T, E, k, H, I = c.T, c.E, c.topk, c.H, c.I
    w1 = [_loop_dequant(p, s, d, H, act) for p, s, d in c.fc1]
    w2 = [_loop_dequant(p, s, d, I, act) for p, s, d in c.fc2]
    for t in range(T):
        logits = [float(v) for v in c.logits[t]]
        order = sorted(range(E), key=lambda e: (-logits[e], e))[:k]
        assert res["idx"][t].tolist() == order
        z = sum(math.exp(logits[e] - logits[order[0]]) for e in order)
        pw = [math.exp(logits[e] - logits[order[0]]) / z for e in order]
        assert np.allclose(res["p"][t], pw, rtol=1e-14)
        x = [float(_VALUE[act](int(b))) for b in c.x_bits[t]]
        acc = [0.0] * H
        for j, e in enumerate(order):
            gate = [math.fsum(x[i] * w1[e][n][i] for i in range(H)) for n in range(I)]
            up = [math.fsum(x[i] * w1[e][I + n][i] for i in range(H)) for n in range(I)]
            h = [float(_VALUE[act](int(formats.act_bits(gate[n] / (1 + math.exp(-gate[n])) * up[n], act))))
                 for n in range(I)]
            for o in range(H):
                y = math.fsum(h[n] * w2[e][o][n] for n in range(I))
                acc[o] += pw[j] * y
        ref = np.array(acc)
        got = res["out"][t]
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
        assert np.array_equal(res["out_bits"][t], formats.act_bits(ref, act))


@pytest.mark.parametrize("act", ["bf16", "f16"])
def test_single_expert_top1_reduces_to_dense(act):
    _single_expert_check(act)


def _single_expert_check(act):
    c = _tiny_layer(T=5, E=1, topk=1, H=64, I=32, seed=9, act=act)
    fc1 = [(p, s, d, True) for p, s, d in c.fc1]
    fc2 = [(p, s, d, True) for p, s, d in c.fc2]
    res = moe.moe_layer(c.x_bits, c.logits, fc1, fc2, 1, act=act)
    assert np.all(res["p"] == 1.0)
    gu, _ = dense.linear(c.x_bits, *fc1[0], act=act)
    h = formats.act_bits(moe.silu(gu[:, :32]) * gu[:, 32:], act)
    y, yb = dense.linear(h, *fc2[0], act=act)
    assert np.array_equal(res["out"], y) and np.array_equal(res["out_bits"], yb)


def test_planted_gate_up_swap_is_caught(monkeypatch):
    orig = moe.moe_layer

    def swapped(x_bits, logits, fc1, fc2, topk, pqs_bits=None, tokens=None, act="bf16"):
        flipped = []
        for p, s, g, d in fc1:
            half = p.shape[0] // 2
            flipped.append((np.concatenate([p[half:], p[:half]]),
                            np.concatenate([s[half:], s[:half]]), g, d))
        return orig(x_bits, logits, flipped, fc2, topk, pqs_bits, tokens, act)
    monkeypatch.setattr(moe, "moe_layer", swapped)
    with pytest.raises(AssertionError):
        _single_expert_check("bf16")


def test_token_subset_and_awq():
    c = _tiny_layer(T=6, E=4, topk=2, seed=13, awq=True)
    fc1 = [(p, s, d, True) for p, s, d in c.fc1]
    fc2 = [(p, s, d, True) for p, s, d in c.fc2]
    full = moe.moe_layer(c.x_bits, c.logits, fc1, fc2, 2, pqs_bits=c.pqs_bits)
    sub = moe.moe_layer(c.x_bits, c.logits, fc1, fc2, 2, pqs_bits=c.pqs_bits, tokens=[4, 1])
    assert np.array_equal(sub["out"], full["out"][[4, 1]])
    plain = moe.moe_layer(c.x_bits, c.logits, fc1, fc2, 2)
    rel = np.linalg.norm(plain["out"] - full["out"]) / np.linalg.norm(full["out"])
    assert rel > 0.1                       # a dropped AWQ scale is visible
    ones = np.full(c.H, 0x3F80, dtype=np.uint16)
    same = moe.moe_layer(c.x_bits, c.logits, fc1, fc2, 2, pqs_bits=ones)
    assert np.array_equal(same["out"], plain["out"])


def test_zero_tokens():
    c = _tiny_layer(T=0, E=4, topk=2)
    res = moe.moe_layer(c.x_bits, c.logits, [(p, s, d, True) for p, s, d in c.fc1],
                        [(p, s, d, True) for p, s, d in c.fc2], 2)
    assert res["out"].shape == (0, c.H) and res["perm"].size == 0
    assert res["offsets"].tolist() == [0] * (c.E + 1)


# ------------------------------------------------------------ dense MLP ---
def _mlp_case(T=2, H=32, I=16, seed=41, act="bf16", awq=False):
    r = synth.rng(seed)
    fc1 = synth.quantize(synth.normal_weight(r, 2 * I, H))
    fc2 = synth.quantize(synth.normal_weight(r, H, I))
    x = synth.normal_act(r, (T, H), act)
    pqs = synth.awq_scale_bits(r, H, act) if awq else None
    return x, fc1, fc2, pqs


@pytest.mark.parametrize("act,awq", [("bf16", False), ("f16", False), ("bf16", True)])
def test_mlp_against_python_loops(act, awq):
    """Every product and sum by hand: exact-rational weights, math.fsum dot
    products, the SwiGLU and both roundings done element by element."""
    T, H, I = 2, 32, 16
    x_bits, fc1, fc2, pqs = _mlp_case(act=act, awq=awq)
    out, out_bits, h_bits = moe.mlp(x_bits, (*fc1, True), (*fc2, True), pqs_bits=pqs, act=act)
    w1 = _loop_dequant(*fc1, H, act)
    w2 = _loop_dequant(*fc2, I, act)
    for t in range(T):
        xv = [_VALUE[act](int(b)) for b in x_bits[t]]
        if awq:
            xv = [_VALUE[act](_ROUND[act](v * _VALUE[act](int(s)))) for v, s in zip(xv, pqs)]
        x = [float(v) for v in xv]
        gate = [math.fsum(x[i] * w1[n][i] for i in range(H)) for n in range(I)]
        up = [math.fsum(x[i] * w1[I + n][i] for i in range(H)) for n in range(I)]
        h = [int(formats.act_bits(gate[n] / (1 + math.exp(-gate[n])) * up[n], act)) for n in range(I)]
        assert h == [int(b) for b in h_bits[t]]
        hv = [float(_VALUE[act](b)) for b in h]
        y = [math.fsum(hv[n] * w2[o][n] for n in range(I)) for o in range(H)]
        assert np.allclose(out[t], y, rtol=1e-12, atol=1e-12 * max(abs(v) for v in y))
        assert np.array_equal(out_bits[t], formats.act_bits(np.array(y), act))


def test_mlp_is_the_single_expert_layer():
    x_bits, fc1, fc2, _ = _mlp_case(T=5, H=64, I=32, seed=43)
    out, out_bits, _ = moe.mlp(x_bits, (*fc1, True), (*fc2, True))
    logits = np.zeros((5, 1), dtype=np.float32)
    res = moe.moe_layer(x_bits, logits, [(*fc1, True)], [(*fc2, True)], 1)
    assert np.array_equal(res["out"], out) and np.array_equal(res["out_bits"], out_bits)


def test_mlp_planted_gate_up_swap_is_caught():
    x_bits, fc1, fc2, _ = _mlp_case(T=3, seed=44)
    p, s, d = fc1
    half = p.shape[0] // 2
    swapped = (np.concatenate([p[half:], p[:half]]), np.concatenate([s[half:], s[:half]]), d, True)
    a, _, _ = moe.mlp(x_bits, (*fc1, True), (*fc2, True))
    b, _, _ = moe.mlp(x_bits, swapped, (*fc2, True))
    assert np.linalg.norm(a - b) / np.linalg.norm(a) > 0.1


# ------------------------------------------------------------ MoE variants ---
def test_relu2_against_exact():
    from fractions import Fraction
    r = np.random.default_rng(3)
    v = r.standard_normal(200) * 3
    got = moe.relu2(v)
    for a, b in zip(v, got):
        want = Fraction(float(a)) ** 2 if a > 0 else Fraction(0)
        assert abs(Fraction(float(b)) - want) <= want * Fraction(1, 2 ** 52)
    assert moe.relu2(np.array([-0.0, 0.0, -5.0]))[2] == 0.0


def _variant_layer(activation, split=False, T=3, E=4, topk=2, H=32, I=16, seed=51, act="bf16"):
    r = synth.rng(seed)
    fc1, fc2 = [], []
    for _ in range(E):
        if activation == "swiglu" and split:
            fc1.append((synth.quantize(synth.normal_weight(r, I, H)), synth.quantize(synth.normal_weight(r, I, H))))
        elif activation == "swiglu":
            fc1.append(synth.quantize(synth.normal_weight(r, 2 * I, H)))
        else:
            fc1.append(synth.quantize(synth.normal_weight(r, I, H)))
        fc2.append(synth.quantize(synth.normal_weight(r, H, I)))
    c = synth.moe_case(T, seed, E=E, topk=topk, H=H, I=I, weights=(fc1, fc2), act=act)
    return c, fc1, fc2


@pytest.mark.parametrize("activation", ["relu2", "silu"])
def test_non_gated_layer_against_python_loops(activation):
    c, fc1, fc2 = _variant_layer(activation)
    T, E, k, H, I = c.T, c.E, c.topk, c.H, c.I
    res = moe.moe_layer(c.x_bits, c.logits, [(p, s, d, True) for p, s, d in fc1],
                        [(p, s, d, True) for p, s, d in fc2], k, activation=activation)
    w1 = [_loop_dequant(p, s, d, H) for p, s, d in fc1]
    w2 = [_loop_dequant(p, s, d, I) for p, s, d in fc2]
    for t in range(T):
        order = res["idx"][t].tolist()
        pw = res["p"][t]
        x = [float(bf16_exact(int(b))) for b in c.x_bits[t]]
        acc = [0.0] * H
        for j, e in enumerate(order):
            v = [math.fsum(x[i] * w1[e][n][i] for i in range(H)) for n in range(I)]
            a = [max(u, 0.0) ** 2 if activation == "relu2" else u / (1 + math.exp(-u)) for u in v]
            h = [float(bf16_exact(int(formats.bf16_bits(u)))) for u in a]
            for o in range(H):
                acc[o] += pw[j] * math.fsum(h[n] * w2[e][o][n] for n in range(I))
        ref = np.array(acc)
        assert np.allclose(res["out"][t], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
        assert np.array_equal(res["out_bits"][t], formats.bf16_bits(ref))


def test_split_gate_up_with_equal_globals_is_the_fused_layer():
    """Gate and up quantized with one shared divisor and stored as two shards give
    exactly the fused [2I, H] layer."""
    c, fc1, fc2 = _variant_layer("swiglu", seed=52)
    I = c.I
    split = [((p[:I], s[:I], d, True), (p[I:], s[I:], d, True)) for p, s, d in fc1]
    fused = moe.moe_layer(c.x_bits, c.logits, [(p, s, d, True) for p, s, d in fc1],
                          [(p, s, d, True) for p, s, d in fc2], c.topk)
    shards = moe.moe_layer(c.x_bits, c.logits, split, [(p, s, d, True) for p, s, d in fc2], c.topk, fc1_split=True)
    assert np.array_equal(fused["out_bits"], shards["out_bits"])


def test_split_gate_up_own_globals_against_python_loops():
    c, fc1, fc2 = _variant_layer("swiglu", split=True, seed=53)
    T, k, H, I = c.T, c.topk, c.H, c.I
    res = moe.moe_layer(c.x_bits, c.logits, [((gp, gs, gd, True), (up, us, ud, True)) for (gp, gs, gd), (up, us, ud) in fc1],
                        [(p, s, d, True) for p, s, d in fc2], k, fc1_split=True)
    assert any(g[2] != u[2] for g, u in fc1)                    # the shards' globals differ
    for t in range(T):
        order = res["idx"][t].tolist()
        x = [float(bf16_exact(int(b))) for b in c.x_bits[t]]
        acc = [0.0] * H
        for j, e in enumerate(order):
            wg = _loop_dequant(*fc1[e][0], H)
            wu = _loop_dequant(*fc1[e][1], H)
            w2 = _loop_dequant(*fc2[e], I)
            gate = [math.fsum(x[i] * wg[n][i] for i in range(H)) for n in range(I)]
            up = [math.fsum(x[i] * wu[n][i] for i in range(H)) for n in range(I)]
            h = [float(bf16_exact(int(formats.bf16_bits(gate[n] / (1 + math.exp(-gate[n])) * up[n])))) for n in range(I)]
            for o in range(H):
                acc[o] += res["p"][t][j] * math.fsum(h[n] * w2[o][n] for n in range(I))
        ref = np.array(acc)
        assert np.array_equal(res["out_bits"][t], formats.bf16_bits(ref))


@pytest.mark.parametrize("act", ["bf16", "f16"])
def test_finalize_pre_quant_scale(act):
    r = synth.rng(61)
    E, H = 5, 48
    w1 = np.stack([synth.awq_scale_bits(r, H, act) for _ in range(E)])
    w3 = np.stack([synth.awq_scale_bits(r, H, act) for _ in range(E)])
    got = moe.finalize_pre_quant_scale(w1, w3, act)
    val = _VALUE[act]
    for k in range(H):
        best = max([val(int(w1[e, k])) for e in range(E)] + [val(int(w3[e, k])) for e in range(E)])
        assert val(int(got[k])) == best
    # one expert: the elementwise max(w3, w1)
    one = moe.finalize_pre_quant_scale(w1[:1], w3[:1], act)
    assert all(val(int(one[k])) == max(val(int(w1[0, k])), val(int(w3[0, k]))) for k in range(H))
