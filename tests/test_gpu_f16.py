"""GPU parity of the FP16-activation path (W4A16 with FP16 activations) against
the CPU oracle: the weight dequantized to FP16 bit for bit, and the GEMM and MoE
outputs within the parity bar against the oracle's FP16-rounded output.  The
same kernels run with FP16 tensor-core MMAs and the FP16 magnitude table."""

import numpy as np
import pytest
import torch

import w4a16_nvfp4_weight_gb300 as nv
from oracle import dense, formats
from oracle import moe as omoe
from tests import gpu_util as gu
from w4a16_nvfp4_weight_gb300 import synth

pytestmark = pytest.mark.gpu
F16 = "f16"


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    torch.cuda.init()
    yield


@pytest.mark.parametrize("divisor,is_div", [(448.0, True), (24366.764, True), (1.0e-3, True),
                                            (1.0e6, True), (-0.37, False)])
def test_dequant_f16_bit_exact_every_scale_code(divisor, is_div):
    """All 256 scale codes x all 16 codes, including FP16 overflow to infinity
    (divisor 1e-3) and FP16 subnormal weights (divisor 1e6)."""
    N, K = 256, 64
    codes = np.tile(np.arange(16, dtype=np.uint8), (N, K // 16))
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    scales = np.repeat(np.arange(256, dtype=np.uint8)[:, None], K // 16, axis=1)
    w = nv.repack(gu.u8(packed), gu.u8(scales), divisor, N, K, global_is_divisor=is_div)
    got = gu.tensor_to_bits(nv.dequant(w, dtype=torch.float16))
    gu.check_device_status()
    want = dense.dequant(packed, scales, divisor, is_div, K, act=F16)
    assert np.array_equal(got, want)
    # the BF16 table of the same buffer is untouched
    got_b = gu.tensor_to_bits(nv.dequant(w))
    assert np.array_equal(got_b, dense.dequant(packed, scales, divisor, is_div, K))


@pytest.mark.parametrize("K,N", [(2064, 1000), (720, 3000), (48, 17)])
def test_dequant_f16_tails(K, N):
    c = synth.gaussian_case(1, K, N, seed=200 + K + N, act=F16)
    w = gu.repack_case(c)
    got = gu.tensor_to_bits(nv.dequant(w, dtype=torch.float16))
    assert np.array_equal(got, dense.dequant(c.packed, c.scales, c.divisor, True, K, act=F16))


def _gemm(c, awq=True):
    w = gu.repack_case(c)
    x = gu.bits_to_tensor(c.x_bits, F16)
    pqs = gu.bits_to_tensor(c.pqs_bits, F16) if (awq and c.pqs_bits is not None) else None
    y = nv.gemm(x, w, pre_quant_scale=pqs)
    gu.check_device_status()
    assert y.dtype == torch.float16
    return gu.tensor_to_bits(y)


@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
@pytest.mark.parametrize("K,N", [(256, 256), (2064, 1000), (720, 3000)])
def test_gemm_f16_decode(M, K, N):
    c = synth.gaussian_case(M, K, N, seed=5000 + 7 * M + K + N, awq=(M % 3 == 0), act=F16)
    _, ref = gu.oracle_linear(c, act=F16)
    gu.compare(_gemm(c), ref, f"f16 M={M} K={K} N={N}", act=F16)


@pytest.mark.parametrize("M", [1, 16])
def test_gemm_f16_decode_deep_ring(M):
    c = synth.gaussian_case(M, 8240, 1024, seed=5100 + M, act=F16)
    _, ref = gu.oracle_linear(c, act=F16)
    gu.compare(_gemm(c), ref, f"f16 M={M} K=8240", act=F16)


@pytest.mark.parametrize("M,K,N", [(17, 256, 256), (300, 2064, 1000), (128, 720, 3000),
                                   (512, 8192, 512), (516, 4096, 1000)])
def test_gemm_f16_tile(M, K, N):
    """The tcgen05 tile kernel with FP16 operands (kind::f16, F16 format), tails,
    AWQ at M=516 and the split-K reduction at (512, 8192) and (516, 4096)."""
    c = synth.gaussian_case(M, K, N, seed=5200 + M + N, awq=(M == 516), act=F16)
    _, ref = gu.oracle_linear(c, act=F16)
    gu.compare(_gemm(c), ref, f"f16 tile M={M} K={K} N={N}", act=F16)


def test_bf16_entry_on_f16_bits_fails_the_bar():
    """Control: the same FP16 activation bits run through the BF16 entry point
    (read as BF16) are far outside the FP16 oracle's bar."""
    c = synth.gaussian_case(4, 256, 256, seed=77, act=F16)
    w = gu.repack_case(c)
    y = gu.tensor_to_bits(nv.gemm(gu.bits_to_tensor(c.x_bits, "bf16"), w))
    _, ref = gu.oracle_linear(c, act=F16)
    with pytest.raises(AssertionError):
        gu.compare(y, ref, "bf16 entry on f16 bits", act=F16)


@pytest.mark.parametrize("M,K,N", [(1, 4096, 14336), (16, 14336, 4096), (2048, 5120, 13824)])
def test_gemm_f16_full_size_sampled(M, K, N):
    r = synth.rng(synth.seed_for(5, K + N + M))
    packed, scales, d = synth.weight_only(K, N, synth.seed_for(5, K * 7 + N))
    w = nv.repack(gu.u8(packed), gu.u8(scales), float(d), N, K)
    rows = np.unique(np.concatenate([r.choice(N, size=32, replace=False), [0, N - 1]]))
    x_bits = synth.normal_act(r, (M, K), F16)
    y = gu.tensor_to_bits(nv.gemm(gu.bits_to_tensor(x_bits, F16), w))
    gu.check_device_status()
    _, ref = dense.linear(x_bits, packed, scales, d, True, rows=rows, act=F16)
    gu.compare(y[:, rows], ref, f"f16 M={M} K={K} N={N}", act=F16)
    assert np.all(np.isfinite(formats.f16_to_float(y)))


def _device_experts(weights, N, K):
    size = nv.repack_size(N, K)
    buf = torch.empty(len(weights) * size, dtype=torch.uint8, device="cuda")
    for e, (p, s, d) in enumerate(weights):
        nv.repack(gu.u8(p), gu.u8(s), float(d), N, K, out=buf[e * size:(e + 1) * size])
    return buf


# (3,4,2,64,64) and (64,16,4,256,128): streaming path; (300,8,2,256,256): tile path
@pytest.mark.parametrize("T,E,topk,H,I,awq", [(3, 4, 2, 64, 64, False), (64, 16, 4, 256, 128, True),
                                              (300, 8, 2, 256, 256, True)])
def test_moe_f16(T, E, topk, H, I, awq):
    r = synth.rng(T + 991)
    fc1 = [synth.quantize(synth.normal_weight(r, 2 * I, H)) for _ in range(E)]
    fc2 = [synth.quantize(synth.normal_weight(r, H, I)) for _ in range(E)]
    c = synth.moe_case(T, T + 3, E=E, topk=topk, H=H, I=I, weights=(fc1, fc2), awq=awq, act=F16)
    x = gu.bits_to_tensor(c.x_bits, F16)
    logits = torch.from_numpy(np.ascontiguousarray(c.logits)).cuda()
    pqs = gu.bits_to_tensor(c.pqs_bits, F16) if awq else None
    out, routing = nv.moe_grouped(x, logits, _device_experts(fc1, 2 * I, H), _device_experts(fc2, H, I),
                                  topk, I, fc1_pre_quant_scale=pqs, return_routing=True)
    gu.check_device_status()
    assert out.dtype == torch.float16
    ref = omoe.moe_layer(c.x_bits, c.logits, [(p, s, d, True) for p, s, d in fc1],
                         [(p, s, d, True) for p, s, d in fc2], topk,
                         pqs_bits=c.pqs_bits if awq else None, act=F16)
    assert np.array_equal(routing["idx"].cpu().numpy().reshape(T, topk), ref["idx"])
    assert np.array_equal(routing["perm"].cpu().numpy(), ref["perm"])
    gu.compare(gu.tensor_to_bits(out), ref["out_bits"], f"f16 MoE T={T}", act=F16)
