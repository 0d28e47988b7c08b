"""W4A16 NVFP4 mixture-of-experts layer, the plain way (test infrastructure).

What the method computes ("[TRTLLM-12288][feat] Support Nemotron-H nvfp4 ckpt
on Hopper", Changes table, MoE row): the weights of the ACTIVE experts are
dequantized to BF16 and a BF16 fused MoE runs on them with empty scales; the
FC1 tensor is the fused gate/up projection ``w3_w1`` and FC2 is ``w2``; gated
experts apply SwiGLU (SGLang PR 40022, review thread on ``is_gated``).  An AWQ
pre-quant scale, when the checkpoint has one, multiplies the BF16 activation
before FC1 ("[None][fix] Apply the NVFP4_AWQ pre-quant scale in MegaMoE
CuteDSL", commit applying the scale on the CUTLASS W4A16 MoE path).  The pages
give no routing arithmetic; the layer's definition is: router logits ->
softmax -> top-k -> renormalise, which is the same as a softmax over the k
selected logits.

Readings taken where the pages are silent:

* top-k is chosen on the FP32 logits; equal logits go to the lower expert
  index; the k output slots are in descending-logit order.
* p[t, j] = exp(l_j - l_max) / sum_{i in top-k} exp(l_i - l_max)  (float64).
* FC1 rows [0, I) are the gate half and rows [I, 2I) the up half.
* h = RN_bf16(silu(gate) * up), silu(v) = v / (1 + exp(-v)), from the exact
  (float64) FC1 outputs; h is FC2's BF16 activation.
* out[t] = RN_bf16( sum_j p[t, j] * y[t, j] ), summed in slot order.
* permutation tables: counts[e], offsets = exclusive scan (E+1 entries),
  perm = the flat routing slots t*k + j sorted stably by expert (so by
  expert, then token, then slot), inv[perm[i]] = i.

With FP16 activations (``act="f16"``; W4A16 covers them: "[TRTLLM-12720]
[feat] Support nvfp4 w4a16 on sm120", Summary) the expert weights, h and the
output are rounded to FP16 instead of BF16.

Parity: pinned by tests/test_oracle_moe.py (hand-built logits with a known
top-k and ties, sum(p) == 1, permutation invariants, E=1/top-1 reduction to the
dense oracle, and a pure-Python loop implementation on a tiny layer).
"""

import numpy as np

from .dense import awq_scale_activation, dequant
from .formats import act_bits, act_to_float


def route(logits, topk):
    """Top-k routing.  Returns (idx int32 [T, topk], p float64 [T, topk])."""
    l = np.asarray(logits, dtype=np.float32)
    T, E = l.shape
    idx = np.empty((T, topk), dtype=np.int32)
    p = np.empty((T, topk), dtype=np.float64)
    experts = np.arange(E)
    for t in range(T):
        # primary key: logit descending; secondary: expert index ascending
        order = np.lexsort((experts, -l[t].astype(np.float64)))
        sel = order[:topk]
        idx[t] = sel
        ls = l[t, sel].astype(np.float64)
        w = np.exp(ls - ls.max())
        p[t] = w / w.sum()
    return idx, p


def permute(idx, E):
    """Permutation tables for grouping routed slots by expert.

    Returns (counts int32 [E], offsets int32 [E+1], perm int32 [T*k],
    inv int32 [T*k]).
    """
    flat = np.asarray(idx, dtype=np.int64).ravel()
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size, dtype=np.int32)
    return counts, offsets, perm, inv


def silu(v):
    return v / (1.0 + np.exp(-v))


def relu2(v):
    """Squared ReLU, max(v, 0)**2: the "relu2" activation of non-gated experts
    (SGLang PR 40022, review thread: relu2 and silu non-gated experts)."""
    r = np.maximum(v, 0.0)
    return r * r


ACTIVATIONS = ("swiglu", "relu2", "silu")


def finalize_pre_quant_scale(w1_pqs_bits, w3_pqs_bits, act="bf16"):
    """The layer's FC1 activation scale from per-expert AWQ pre-quant scales:
    s[k] = max over experts e of max(w3_e[k], w1_e[k]) ("[None][fix] Apply the
    NVFP4_AWQ pre-quant scale in MegaMoE CuteDSL", Description, step 2: the
    finalization writes max(w3, w1) into the [1, hidden] FC1 input scale).
    Inputs uint16 [E, H] bit patterns of the activation type; returns uint16 [H]."""
    a = act_to_float(np.asarray(w1_pqs_bits, dtype=np.uint16), act)
    b = act_to_float(np.asarray(w3_pqs_bits, dtype=np.uint16), act)
    return act_bits(np.maximum(a, b).max(axis=0), act)


def expert_weights(fc, K, act="bf16"):
    """Dequantized weight values (float64) of one expert matrix, rounded to the
    activation type.

    ``fc`` = (packed, scales, global_scale, global_is_divisor).
    """
    packed, scales, gs, is_div = fc
    return act_to_float(dequant(packed, scales, gs, is_div, K, act), act)


def _fc1_out(x, fc1_e, H, act, activation, fc1_split):
    """h (bit patterns) of one expert for the rows x (float64), and I."""
    if activation == "swiglu":
        if fc1_split:      # gate and up quantized separately, each with its own global
            w1 = np.concatenate([expert_weights(fc1_e[0], H, act), expert_weights(fc1_e[1], H, act)])
        else:
            w1 = expert_weights(fc1_e, H, act)
        I = w1.shape[0] // 2
        gu = x @ w1.T
        return act_bits(silu(gu[:, :I]) * gu[:, I:], act)
    w1 = expert_weights(fc1_e, H, act)                  # non-gated: [I, H]
    v = x @ w1.T
    if activation == "relu2":
        return act_bits(relu2(v), act)
    if activation == "silu":
        return act_bits(silu(v), act)
    raise ValueError(f"unknown activation {activation!r}")


def moe_layer(x_bits, logits, fc1, fc2, topk, pqs_bits=None, tokens=None, act="bf16", activation="swiglu",
              fc1_split=False):
    """The whole layer.

    x_bits  uint16 [T, H] activations (BF16, or FP16 with act="f16")
    logits  float32 [T, E] router logits
    fc1     list of E tuples (packed [2I, H/2], scales [2I, H/16], global, is_divisor);
            with fc1_split, E pairs (gate tuple [I, H], up tuple [I, H]), each
            with its own global (per-shard w1/w3 globals, SGLang PR 40022,
            review thread: per-shard global/input scales); with a non-gated
            activation ("relu2" or "silu"), E tuples of [I, H]
    fc2     list of E tuples (packed [H, I/2], scales [H, I/16], global, is_divisor)
    tokens  optional subset of token indices whose outputs are computed
            (routing and permutation tables are always computed for all T)

    Returns a dict with idx, p, counts, offsets, perm, inv, and for the
    computed tokens: out (float64 [T', H]), out_bits (uint16 [T', H]),
    h_bits (uint16 [T', topk, I]) and the token list.
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    T, H = x_bits.shape
    E = len(fc1)
    idx, p = route(logits, topk)
    counts, offsets, perm, inv = permute(idx, E)
    res = dict(idx=idx, p=p, counts=counts, offsets=offsets, perm=perm, inv=inv)
    if tokens is None:
        tokens = np.arange(T)
    tokens = np.asarray(tokens, dtype=np.int64)
    res["tokens"] = tokens
    if T == 0 or tokens.size == 0:
        res["out"] = np.zeros((0, H))
        res["out_bits"] = np.zeros((0, H), dtype=np.uint16)
        return res
    xs = x_bits[tokens]
    if pqs_bits is not None:
        xs = awq_scale_activation(xs, pqs_bits, act)
    x = act_to_float(xs, act)
    if activation == "swiglu":
        I = np.asarray(fc1[0][0][0] if fc1_split else fc1[0][0]).shape[0] // (1 if fc1_split else 2)
    else:
        I = np.asarray(fc1[0][0]).shape[0]
    y = np.zeros((tokens.size, topk, H))
    h_all = np.zeros((tokens.size, topk, I), dtype=np.uint16)
    sel = idx[tokens]                                   # [T', topk]
    for e in np.unique(sel):
        rows, slots = np.nonzero(sel == e)
        w2 = expert_weights(fc2[e], I, act)             # [H, I]
        h = _fc1_out(x[rows], fc1[e], H, act, activation, fc1_split)   # [r, I]
        h_all[rows, slots] = h
        y[rows, slots] = act_to_float(h, act) @ w2.T    # [r, H]
    out = np.zeros((tokens.size, H))
    for j in range(topk):                                # slot order
        out = out + p[tokens, j][:, None] * y[:, j]
    res["out"] = out
    res["out_bits"] = act_bits(out, act)
    res["h_bits"] = h_all
    return res


def mlp(x_bits, fc1, fc2, pqs_bits=None, act="bf16"):
    """Dense gated MLP: the expert computation of ``moe_layer`` on one weight
    pair, for every token (SwiGLU of gated experts: SGLang PR 40022, review
    thread on ``is_gated``; fused gate/up FC1: "[TRTLLM-12288][feat] Support
    Nemotron-H nvfp4 ckpt on Hopper", Changes table).

    fc1 = (packed [2I, H/2], scales [2I, H/16], global, is_divisor), rows
    [0, I) gate and [I, 2I) up; fc2 = (packed [H, I/2], scales [H, I/16],
    global, is_divisor).  Returns (out float64 [T, H], out_bits, h_bits).
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    T, H = x_bits.shape
    I = np.asarray(fc1[0]).shape[0] // 2
    xs = x_bits if pqs_bits is None else awq_scale_activation(x_bits, pqs_bits, act)
    x = act_to_float(xs, act)
    gu = x @ expert_weights(fc1, H, act).T                # [T, 2I], exact float64
    h = act_bits(silu(gu[:, :I]) * gu[:, I:], act)
    out = act_to_float(h, act) @ expert_weights(fc2, I, act).T
    return out, act_bits(out, act), h
