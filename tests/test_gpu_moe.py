"""GPU parity of the grouped top-k MoE layer against the CPU oracle.

Routing indices, the permutation and the per-expert offsets are compared bit
for bit; routing weights to float32 rounding; the layer output within the
parity bar (relative Frobenius <= 2e-3, max-abs <= 2e-2 * max|ref|) against the
oracle's BF16 output.  The full 128-expert layer is checked on sampled tokens.
"""

import numpy as np
import pytest
import torch

import w4a16_nvfp4_weight_gb300 as nv
from oracle import moe as omoe
from tests import gpu_util as gu
from w4a16_nvfp4_weight_gb300 import synth

pytestmark = pytest.mark.gpu


def _device_experts(weights, N, K):
    """Repack E expert matrices back to back into one device buffer."""
    size = nv.repack_size(N, K)
    buf = torch.empty(len(weights) * size, dtype=torch.uint8, device="cuda")
    for e, (p, s, d) in enumerate(weights):
        nv.repack(gu.u8(p), gu.u8(s), float(d), N, K, out=buf[e * size:(e + 1) * size])
    return buf


def _run(c, awq=False):
    fc1 = _device_experts(c.fc1, 2 * c.I, c.H)
    fc2 = _device_experts(c.fc2, c.H, c.I)
    x = gu.bits_to_bf16_tensor(c.x_bits)
    logits = torch.from_numpy(np.ascontiguousarray(c.logits)).cuda()
    pqs = gu.bits_to_bf16_tensor(c.pqs_bits) if awq else None
    out, r = nv.moe_grouped(x, logits, fc1, fc2, c.topk, c.I, fc1_pre_quant_scale=pqs, return_routing=True)
    gu.check_device_status()
    return gu.tensor_to_bits(out), {k: v.cpu().numpy() for k, v in r.items()}


def _oracle(c, awq=False, tokens=None):
    return omoe.moe_layer(c.x_bits, c.logits, [(p, s, d, True) for p, s, d in c.fc1],
                          [(p, s, d, True) for p, s, d in c.fc2], c.topk,
                          pqs_bits=c.pqs_bits if awq else None, tokens=tokens)


def _check_routing(got, ref, T, topk, E):
    assert np.array_equal(got["idx"].reshape(T, topk), ref["idx"])
    assert np.array_equal(got["offsets"], ref["offsets"])
    assert np.array_equal(got["perm"], ref["perm"])
    assert np.allclose(got["p"].reshape(T, topk), ref["p"], rtol=2e-6, atol=1e-7)


def _small_case(T, E, topk, H, I, seed, awq=False):
    r = synth.rng(seed + 77)
    fc1 = [synth.quantize(synth.normal_weight(r, 2 * I, H)) for _ in range(E)]
    fc2 = [synth.quantize(synth.normal_weight(r, H, I)) for _ in range(E)]
    return synth.moe_case(T, seed, E=E, topk=topk, H=H, I=I, weights=(fc1, fc2), awq=awq)


# (300,8,2,256,256), (100,4,3,384,128) and (1024,4,2,128,128) route >= 32 rows per
# expert and take the tensor-core tile path (128- and 256-row items); the others take
# the streaming path ((64,16,4,256,128): 16 rows per expert, some experts in two items).
@pytest.mark.parametrize("T,E,topk,H,I", [(3, 4, 2, 64, 64), (64, 16, 4, 256, 128), (37, 8, 3, 192, 320),
                                          (5, 1, 1, 128, 64), (200, 32, 8, 128, 64), (300, 8, 2, 256, 256),
                                          (100, 4, 3, 384, 128), (1024, 4, 2, 128, 128)])
def test_moe_small_full_compare(T, E, topk, H, I):
    c = _small_case(T, E, topk, H, I, seed=T * 31 + E)
    out, routing = _run(c)
    ref = _oracle(c)
    _check_routing(routing, ref, T, topk, E)
    gu.compare(out, ref["out_bits"], f"MoE T={T} E={E} k={topk}")


@pytest.mark.parametrize("awq", [False, True])
def test_moe_tile_path_expert_tails(awq):
    """Tile path (about 150 rows per expert: 128-row items): expert 0 gets 135
    rows (a 7-row tail past its full tile, run as a streaming item), expert 1
    165 rows (a 37-row tail, more than the 32 a streaming tail takes, so a
    second tile item).  Every output row against the oracle, and with AWQ the
    tail rows are scaled inside the streaming kernel, the others while
    gathering."""
    T, E, topk, H, I = 300, 2, 1, 256, 128
    c = _small_case(T, E, topk, H, I, seed=91, awq=awq)
    logits = np.zeros((T, E), dtype=np.float32)
    logits[:135, 0] = 1.0
    logits[135:, 1] = 1.0
    c.logits = logits
    out, routing = _run(c, awq=awq)
    ref = _oracle(c, awq=awq)
    _check_routing(routing, ref, T, topk, E)
    assert routing["offsets"].tolist() == [0, 135, 300]
    gu.compare(out, ref["out_bits"], f"MoE tile tails awq={awq}")


def test_moe_awq_and_dropped_scale_control():
    c = _small_case(10, 8, 2, 128, 64, seed=5, awq=True)
    out, routing = _run(c, awq=True)
    ref = _oracle(c, awq=True)
    _check_routing(routing, ref, 10, 2, 8)
    gu.compare(out, ref["out_bits"], "MoE AWQ")
    out_plain, _ = _run(c, awq=False)
    with pytest.raises(AssertionError):
        gu.compare(out_plain, ref["out_bits"], "MoE dropped AWQ")


def test_moe_tile_path_awq_and_dropped_scale_control():
    c = _small_case(300, 8, 2, 256, 256, seed=15, awq=True)
    out, routing = _run(c, awq=True)
    ref = _oracle(c, awq=True)
    _check_routing(routing, ref, 300, 2, 8)
    gu.compare(out, ref["out_bits"], "MoE tile path AWQ")
    out_plain, _ = _run(c, awq=False)
    with pytest.raises(AssertionError):
        gu.compare(out_plain, ref["out_bits"], "MoE tile path dropped AWQ")


def test_moe_ties_pick_lower_expert():
    c = _small_case(4, 8, 3, 64, 64, seed=9)
    c.logits[:] = 0.0
    c.logits[1, [5, 2, 7]] = 1.5          # three-way tie at the top
    c.logits[2, :] = -0.0
    out, routing = _run(c)
    ref = _oracle(c)
    _check_routing(routing, ref, 4, 3, 8)
    assert routing["idx"].reshape(4, 3)[1].tolist() == [2, 5, 7]
    gu.compare(out, ref["out_bits"], "MoE ties")


def test_moe_zero_tokens_launch_nothing():
    c = _small_case(0, 4, 2, 64, 64, seed=1)
    fc1 = _device_experts(c.fc1, 128, 64)
    fc2 = _device_experts(c.fc2, 64, 64)
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    logits = torch.empty((0, 4), dtype=torch.float32, device="cuda")
    out = nv.moe_grouped(x, logits, fc1, fc2, 2, 64)
    assert out.shape == (0, 64)
    gu.check_device_status()


def test_moe_deterministic():
    c = _small_case(64, 16, 4, 256, 128, seed=3)
    a, _ = _run(c)
    b, _ = _run(c)
    assert np.array_equal(a, b)


@pytest.fixture(scope="module")
def full_experts():
    """The 128-expert layer: FC1 [1536 x 2048], FC2 [2048 x 768] per expert."""
    E, H, I = 128, 2048, 768
    fc1, fc2 = synth.moe_weights(E, H, I, synth.seed_for(3, 500))
    return E, H, I, fc1, fc2, _device_experts(fc1, 2 * I, H), _device_experts(fc2, H, I)


def _covering_tokens(idx, E, at_least, seed):
    """A seeded token sample whose routed experts cover all E experts (tokens
    are taken in a seeded order when they add an uncovered expert), topped up
    with further seeded tokens to `at_least` (or all tokens)."""
    T = idx.shape[0]
    order = synth.rng(seed).permutation(T)
    chosen, covered = [], set()
    for t in order:
        new = set(int(e) for e in idx[t]) - covered
        if new:
            chosen.append(int(t))
            covered |= new
        if len(covered) == E:
            break
    for t in order:
        if len(chosen) >= min(at_least, T):
            break
        if int(t) not in chosen:
            chosen.append(int(t))
    return sorted(chosen), covered


@pytest.mark.parametrize("T", [1, 16, 256, 4096])
def test_moe_full_size_sampled(full_experts, T):
    """The full layer.  At T = 256 (16 rows per expert: streaming kernels) and
    T = 4096 (256 rows per expert: gathered rows on the tcgen05 tile kernels)
    at least 64 tokens are compared, chosen so that their routing reaches every
    one of the 128 experts, i.e. every expert's FC1 and FC2 work is checked."""
    E, H, I, fc1, fc2, d1, d2 = full_experts
    c = synth.moe_case(T, synth.seed_for(3, T), E=E, topk=8, H=H, I=I, weights=(fc1, fc2))
    x = gu.bits_to_bf16_tensor(c.x_bits)
    logits = torch.from_numpy(np.ascontiguousarray(c.logits)).cuda()
    out, r = nv.moe_grouped(x, logits, d1, d2, 8, I, return_routing=True)
    gu.check_device_status()
    out = gu.tensor_to_bits(out)
    routing = {k: v.cpu().numpy() for k, v in r.items()}
    ref_routing = omoe.route(c.logits, 8)
    if T >= 256:
        tokens, covered = _covering_tokens(ref_routing[0], E, 64, seed=T)
        assert len(covered) == E and len(tokens) >= 64
    else:
        tokens = sorted(set([0, T - 1, T // 2]))
    ref = _oracle(c, tokens=tokens)
    _check_routing(routing, ref, T, 8, E)
    gu.compare(out[tokens], ref["out_bits"], f"MoE T={T} sampled")


@pytest.mark.parametrize("T", [1, 16, 64, 65, 256, 4096])
def test_moe_route_tables_bit_exact(T):
    """The standalone routing call (the fused single-CTA kernel up to 64
    tokens; above, a routing kernel and a single-CTA permutation, since the
    call has no workspace for the layer's chunked kernels) against the oracle:
    top-k indices, the stable permutation, its inverse and the expert offsets
    bit for bit, the routing weights to float32 rounding."""
    E, topk = 128, 8
    c = synth.moe_case(T, synth.seed_for(3, T) + 7, E=E, topk=topk, H=64, I=64, weights=None)
    logits = torch.from_numpy(np.ascontiguousarray(c.logits)).cuda()
    got = {k: v.cpu().numpy() for k, v in nv.moe_route(logits, topk).items()}
    gu.check_device_status()
    idx, p = omoe.route(c.logits, topk)
    counts, offsets, perm, inv = omoe.permute(idx, E)
    assert np.array_equal(got["idx"], idx)
    assert np.allclose(got["p"], p, rtol=2e-6, atol=1e-7)
    assert np.array_equal(got["perm"], perm)
    assert np.array_equal(got["inv"], inv)
    assert np.array_equal(got["offsets"], offsets)
    assert np.array_equal(got["inv"][got["perm"]], np.arange(T * topk))


def test_moe_route_ties_and_negative_zero():
    logits = np.zeros((3, 8), dtype=np.float32)
    logits[0, [6, 1, 4]] = 2.0                 # three-way tie at the top
    logits[1, :] = -0.0
    logits[2, 3] = np.float32(-0.0)
    got = {k: v.cpu().numpy() for k, v in nv.moe_route(torch.from_numpy(logits).cuda(), 3).items()}
    idx, p = omoe.route(logits, 3)
    _, offsets, perm, inv = omoe.permute(idx, 8)
    assert got["idx"][0].tolist() == [1, 4, 6]
    for k, v in (("idx", idx), ("perm", perm), ("inv", inv), ("offsets", offsets)):
        assert np.array_equal(got[k], v), k


@pytest.mark.parametrize("T,E,topk", [(64, 256, 16), (65, 256, 16), (7, 40, 5), (100, 3, 3), (33, 1, 1)])
def test_moe_route_tables_edge_shapes(T, E, topk):
    """Both routing kernels at the edges of their limits: 256 experts with
    top-16 at 64 tokens (the last fused size) and 65 (the first two-kernel
    size), an expert count that is not a multiple of 32, top-k = E, and one
    expert."""
    c = synth.moe_case(T, synth.seed_for(3, T) + E, E=E, topk=topk, H=64, I=64, weights=None)
    got = {k: v.cpu().numpy() for k, v in nv.moe_route(torch.from_numpy(np.ascontiguousarray(c.logits)).cuda(),
                                                         topk).items()}
    gu.check_device_status()
    idx, p = omoe.route(c.logits, topk)
    _, offsets, perm, inv = omoe.permute(idx, E)
    for k, v in (("idx", idx), ("perm", perm), ("inv", inv), ("offsets", offsets)):
        assert np.array_equal(got[k], v), k
    assert np.allclose(got["p"], p, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("T,E,topk", [(513, 256, 16), (530, 40, 5), (600, 3, 3), (803, 1, 1), (4097, 128, 8),
                                       (65, 256, 16), (130, 40, 5)])
def test_moe_layer_chunked_routing_tables(T, E, topk):
    """From 513 tokens the layer routes and permutes in chunks of 8 tokens (a
    CTA per chunk: routing + per-expert counts; a scan of each expert's counts
    over the chunks; each chunk's positions after the earlier chunks'); from
    65 to 512 a routing kernel and a single-CTA permutation: 256 experts with
    top-16, an expert count that is not a multiple of 32, top-k = E, one
    expert and ragged last chunks -- indices, the stable permutation and the
    offsets bit for bit against the oracle, and the layer output on a few
    tokens."""
    H = I = 64
    c = _small_case(T, E, topk, H, I, seed=T + E)
    out, routing = _run(c)
    tokens = sorted(set([0, 1, T // 2, T - 1]))
    ref = _oracle(c, tokens=tokens)
    _check_routing(routing, ref, T, topk, E)
    _, offsets, perm, inv = omoe.permute(ref["idx"], E)
    assert np.array_equal(routing["perm"], perm)
    gu.compare(out[tokens], ref["out_bits"], f"MoE T={T} E={E} top-{topk}")


@pytest.mark.parametrize("T", [5, 70])
def test_moe_route_nan_and_infinite_logits(T):
    """NaN logits rank below every number (a sort that puts NaN last, ties to
    the lower expert index) and infinities are ordinary extremes; fused
    (T <= 64) and two-kernel routing."""
    E, topk = 16, 4
    r = synth.rng(T + 1)
    logits = r.standard_normal((T, E)).astype(np.float32)
    logits[:, 3] = np.nan
    logits[::2, 9] = np.nan
    logits[1, 12] = np.inf
    logits[2, :] = -np.inf
    logits[2, 5] = np.nan
    logits[3, :] = np.nan                          # every logit NaN: experts 0..3
    got = {k: v.cpu().numpy() for k, v in nv.moe_route(torch.from_numpy(logits).cuda(), topk).items()}
    idx, p = omoe.route(logits, topk)
    _, offsets, perm, inv = omoe.permute(idx, E)
    for k, v in (("idx", idx), ("perm", perm), ("inv", inv), ("offsets", offsets)):
        assert np.array_equal(got[k], v), k
    assert got["idx"][3].tolist() == [0, 1, 2, 3]
    finite = np.isfinite(p).all(axis=1)
    assert np.allclose(got["p"][finite], p[finite], rtol=2e-6, atol=1e-7)
