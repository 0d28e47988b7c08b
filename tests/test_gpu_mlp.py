"""GPU parity of the dense gated MLP (FC1 gate/up + SwiGLU on the MoE FC1
kernels, FC2 on the dense GEMM) against the CPU oracle, within the parity bar:
the streaming FC1 kernel (few tokens), the tcgen05 FC1 tiles (many tokens),
AWQ, FP16 activations, T = 0, and a Llama-sized layer on sampled outputs."""

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


def _weights(H, I, seed):
    r = synth.rng(seed)
    return synth.quantize(synth.normal_weight(r, 2 * I, H)), synth.quantize(synth.normal_weight(r, H, I))


def _repack(w, N, K):
    p, s, d = w
    return nv.repack(gu.u8(p), gu.u8(s), float(d), N, K)


# T <= 16 and small tile grids: streaming FC1; (600, 256, 256) and (520, 512, 128): tile FC1
@pytest.mark.parametrize("T,H,I,act,awq", [(1, 128, 64, "bf16", False), (13, 192, 320, "bf16", True),
                                           (16, 256, 128, "f16", False), (40, 256, 192, "bf16", False),
                                           (600, 256, 256, "bf16", True), (520, 512, 128, "f16", True)])
def test_mlp_parity(T, H, I, act, awq):
    fc1, fc2 = _weights(H, I, seed=T + H + I)
    r = synth.rng(T * 7 + I)
    x = synth.normal_act(r, (T, H), act)
    pqs = synth.awq_scale_bits(r, H, act) if awq else None
    out = nv.mlp(gu.bits_to_tensor(x, act), _repack(fc1, 2 * I, H), _repack(fc2, H, I),
                 fc1_pre_quant_scale=gu.bits_to_tensor(pqs, act) if awq else None)
    gu.check_device_status()
    _, ref, _ = omoe.mlp(x, (*fc1, True), (*fc2, True), pqs_bits=pqs, act=act)
    gu.compare(gu.tensor_to_bits(out), ref, f"MLP T={T} H={H} I={I} {act} awq={awq}", act=act)


def test_mlp_dropped_awq_scale_fails_the_bar():
    fc1, fc2 = _weights(128, 64, seed=5)
    r = synth.rng(6)
    x = synth.normal_act(r, (8, 128), "bf16")
    pqs = synth.awq_scale_bits(r, 128)
    out = nv.mlp(gu.bits_to_tensor(x, "bf16"), _repack(fc1, 128, 128), _repack(fc2, 128, 64))
    _, ref, _ = omoe.mlp(x, (*fc1, True), (*fc2, True), pqs_bits=pqs)
    with pytest.raises(AssertionError):
        gu.compare(gu.tensor_to_bits(out), ref, "MLP dropped AWQ")


def test_mlp_zero_tokens():
    fc1, fc2 = _weights(128, 64, seed=7)
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    out = nv.mlp(x, _repack(fc1, 128, 128), _repack(fc2, 128, 64))
    assert out.shape == (0, 128)
    gu.check_device_status()


def test_mlp_llama_size_sampled():
    """H = 4096, I = 14336 (FC1 [28672, 4096], FC2 [4096, 14336]) at T = 1, 16
    and 512 on sampled tokens, checked against one oracle call."""
    H, I = 4096, 14336
    fc1, fc2 = _weights(H, I, seed=11)
    w1, w2 = _repack(fc1, 2 * I, H), _repack(fc2, H, I)
    xs, outs = [], []
    for T in (1, 16, 512):
        x = synth.normal_act(synth.rng(12 + T), (T, H), "bf16")
        out = gu.tensor_to_bits(nv.mlp(gu.bits_to_tensor(x, "bf16"), w1, w2))
        gu.check_device_status()
        tokens = sorted(set([0, T // 2, T - 1]))
        xs.append(x[tokens])
        outs.append(out[tokens])
    _, ref, _ = omoe.mlp(np.concatenate(xs), (*fc1, True), (*fc2, True))
    gu.compare(np.concatenate(outs), ref, "MLP 4096x14336 T=1,16,512 sampled")
