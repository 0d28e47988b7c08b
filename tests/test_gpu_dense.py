"""GPU parity of the dense path (repack, dequant, GEMM) against the CPU oracle.

Dequantized weights are compared bit for bit; GEMM outputs within the parity
bar (relative Frobenius <= 2e-3, max-abs <= 2e-2 * max|ref|) against the
oracle's BF16-rounded output.  Small cases are checked element by element;
the full workload sizes on sampled output features.
"""

import numpy as np
import pytest
import torch

import w4a16_nvfp4_weight_gb300 as nv
from oracle import dense, formats
from tests import gpu_util as gu
from w4a16_nvfp4_weight_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(lib):
    torch.cuda.init()
    yield


def _unrepack(buf, N, K):
    """Recover checkpoint codes/scales from the repacked bytes, following the
    layout documented in include/nvfp4_w4a16.h."""
    b = np.asarray(buf, dtype=np.uint8)
    hdr = b[:256]
    assert int(hdr[:4].view(np.uint32)[0]) == 0x34504E56
    Np, Kp = -(-N // 256) * 256, -(-K // 64) * 64
    KB = Kp // 64
    sign_pos = [7, 15, 23, 31, 3, 11, 19, 27]
    codes = np.zeros((Np, Kp), dtype=np.uint8)
    scales = np.zeros((Np, Kp // 16), dtype=np.uint8)
    atoms = b[8448:8448 + (Np // 16) * KB * 576].reshape(Np // 256, KB, 16, 576)
    for lane in range(32):
        r, q = lane // 4, lane % 4
        words = atoms[:, :, :, 16 * lane:16 * lane + 16].copy().view(np.uint32)  # [nt,KB,16,4]
        sc = atoms[:, :, :, 512 + 2 * lane:512 + 2 * lane + 2]
        for h in range(2):
            rows = (np.arange(Np // 256)[:, None, None] * 256 + np.arange(16)[None, None, :] * 16 + r + 8 * h)
            for wi in range(2):
                w = words[:, :, :, 2 * h + wi]
                for i in range(8):
                    mag = (w >> (4 * i)) & 7
                    sgn = (w >> sign_pos[i]) & 1
                    kk = np.arange(KB)[None, :, None] * 64 + q * 16 + wi * 8 + i
                    codes[np.broadcast_to(rows, mag.shape), np.broadcast_to(kk, mag.shape)] = (mag | (sgn << 3)).astype(np.uint8)
            kg = np.arange(KB)[None, :, None] * 4 + q
            scales[np.broadcast_to(rows, sc[..., h].shape), np.broadcast_to(kg, sc[..., h].shape)] = sc[..., h]
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed[:N, :K // 2], scales[:N, :K // 16], codes, scales


def test_repack_layout_and_determinism():
    c = synth.gaussian_case(1, 720, 300, seed=7)
    w1 = gu.repack_case(c)
    w2 = gu.repack_case(c)
    torch.cuda.synchronize()
    b1, b2 = w1.buf.cpu().numpy(), w2.buf.cpu().numpy()
    assert np.array_equal(b1, b2)
    packed, scales, codes_pad, scales_pad = _unrepack(b1, c.N, c.K)
    assert np.array_equal(packed, c.packed)
    assert np.array_equal(scales, c.scales)
    assert not codes_pad[c.N:].any() and not codes_pad[:, c.K:].any()
    assert not scales_pad[c.N:].any() and not scales_pad[:, c.K // 16:].any()
    g = np.frombuffer(b1[40:44].tobytes(), dtype=np.float32)[0]
    assert g == np.float32(1.0) / np.float32(c.divisor)


def _dequant_gpu(case):
    w = gu.repack_case(case)
    out = nv.dequant(w)
    gu.check_device_status()
    return gu.tensor_to_bits(out)


def test_dequant_bit_exact_uniform_codes():
    c = synth.uniform_codes_case()
    got = _dequant_gpu(c)
    want = dense.dequant(c.packed, c.scales, c.divisor, True, c.K)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("divisor,is_div", [(448.0, True), (3.0, True), (24366.764, True),
                                            (1.0, False), (-0.37, False), (1.0e-30, True)])
def test_dequant_bit_exact_every_scale_code(divisor, is_div):
    """All 256 scale codes (negative, subnormal and NaN included) x all 16 codes."""
    N, K = 256, 64
    codes = np.tile(np.arange(16, dtype=np.uint8), (N, K // 16))
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    scales = np.repeat(np.arange(256, dtype=np.uint8)[:, None], K // 16, axis=1)
    w = nv.repack(gu.u8(packed), gu.u8(scales), divisor, N, K, global_is_divisor=is_div)
    got = gu.tensor_to_bits(nv.dequant(w))
    gu.check_device_status()
    want = dense.dequant(packed, scales, divisor, is_div, K)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("K,N", [(2064, 1000), (720, 3000), (16, 1), (48, 17), (4096, 512)])
def test_dequant_bit_exact_tails(K, N):
    c = synth.gaussian_case(1, K, N, seed=100 + K + N)
    got = _dequant_gpu(c)
    want = dense.dequant(c.packed, c.scales, c.divisor, True, c.K)
    assert np.array_equal(got, want)


def _gemm(case, awq=True):
    w = gu.repack_case(case)
    x = gu.bits_to_bf16_tensor(case.x_bits)
    pqs = gu.bits_to_bf16_tensor(case.pqs_bits) if (awq and case.pqs_bits is not None) else None
    y = nv.gemm(x, w, pre_quant_scale=pqs)
    gu.check_device_status()
    return gu.tensor_to_bits(y)


def test_gemm_uniform_codes_4x256x256():
    c = synth.uniform_codes_case()
    y = _gemm(c)
    _, ref = gu.oracle_linear(c)
    gu.compare(y, ref, "4x256x256")


@pytest.mark.parametrize("M", list(range(1, 17)))
@pytest.mark.parametrize("K,N", [(256, 256), (2064, 1000), (720, 3000), (1024, 384)])
def test_gemm_decode_small(M, K, N):
    c = synth.gaussian_case(M, K, N, seed=1000 + 7 * M + K + N, awq=(M % 3 == 0))
    y = _gemm(c)
    _, ref = gu.oracle_linear(c)
    gu.compare(y, ref, f"M={M} K={K} N={N}")


@pytest.mark.parametrize("M", [1, 9, 16])
def test_gemm_decode_deep_ring_partial_stages(M):
    """K = 8240 over 8 splits: 17-block slices (long enough for the deep ring)
    whose last ring stage holds one block, a last split of 10 blocks and a
    48-element K tail; 64 CTAs, so the grid is spread one per SM."""
    c = synth.gaussian_case(M, 8240, 1024, seed=4000 + M, awq=(M == 9))
    y = _gemm(c)
    _, ref = gu.oracle_linear(c)
    gu.compare(y, ref, f"M={M} K=8240 N=1024")


@pytest.mark.parametrize("M", [17, 100, 128, 300])
@pytest.mark.parametrize("K,N", [(256, 256), (2064, 1000), (720, 3000)])
def test_gemm_larger_m_small(M, K, N):
    c = synth.gaussian_case(M, K, N, seed=2000 + M + K + N, awq=(M == 100))
    y = _gemm(c)
    _, ref = gu.oracle_linear(c)
    gu.compare(y, ref, f"M={M} K={K} N={N}")


@pytest.mark.parametrize("M,K,N", [(512, 8192, 512), (516, 4096, 1000), (600, 6144, 384)])
def test_gemm_tile_split_k(M, K, N):
    """Few output tiles and a long K: the tile kernel splits K and sums the FP32
    partials in split order (M and N tails included)."""
    c = synth.gaussian_case(M, K, N, seed=3000 + M + N, awq=(M == 516))
    y = _gemm(c)
    _, ref = gu.oracle_linear(c)
    gu.compare(y, ref, f"split-K M={M} K={K} N={N}")
    y2 = _gemm(c)
    assert np.array_equal(y, y2)          # fixed reduction order


def test_dropped_awq_scale_fails_the_bar():
    c = synth.gaussian_case(8, 1024, 512, seed=77, awq=True)
    y_no = _gemm(c, awq=False)
    _, ref = gu.oracle_linear(c, awq=True)
    with pytest.raises(AssertionError):
        gu.compare(y_no, ref, "dropped AWQ")


def test_zero_rows_launch_nothing():
    c = synth.gaussian_case(1, 256, 256, seed=5)
    w = gu.repack_case(c)
    y = torch.full((0, 256), 1.0, dtype=torch.bfloat16, device="cuda")
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    nv.gemm(x, w, out=y)
    gu.check_device_status()


def test_mismatched_header_is_reported_not_trapped():
    c = synth.gaussian_case(2, 256, 256, seed=6)
    w = gu.repack_case(c)
    bad = nv.NVFP4Weight(w.buf, 128, 256)          # header says N=256
    x = gu.bits_to_bf16_tensor(c.x_bits)
    y = torch.full((2, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    nv.gemm(x, bad, out=y)
    assert nv.device_status(clear=True) == 7
    assert torch.all(y == 3.0)
    gu.check_device_status()


@pytest.mark.parametrize("M,K,N_hdr,N_claim", [(600, 256, 256, 128), (1000, 1024, 20480, 20224)])
def test_mismatched_header_tile_kernels(M, K, N_hdr, N_claim):
    """The same header check on the two tile kernels (the tensor-memory-A kernel
    at 600x256, the shared-memory one at 1000x1024): status 7, Y untouched."""
    packed, scales, d = synth.weight_only(K, N_hdr, 12)
    w = nv.repack(gu.u8(packed), gu.u8(scales), float(d), N_hdr, K)
    bad = nv.NVFP4Weight(w.buf, N_claim, K)
    x = gu.bits_to_bf16_tensor(synth.normal_bf16(synth.rng(13), (M, K)))
    y = torch.full((M, N_claim), 3.0, dtype=torch.bfloat16, device="cuda")
    nv.gemm(x, bad, out=y)
    assert nv.device_status(clear=True) == 7
    assert torch.all(y == 3.0)
    gu.check_device_status()


def _sampled_rows(N, r, n=48):
    rows = np.unique(np.concatenate([r.choice(N, size=n, replace=False), [0, N - 1]]))
    return rows


@pytest.mark.parametrize("K,N", [(4096, 4096), (4096, 14336), (14336, 4096), (5120, 25600)])
def test_gemm_decode_full_size_sampled(K, N):
    r = synth.rng(synth.seed_for(1, K + N))
    packed, scales, d = synth.weight_only(K, N, synth.seed_for(1, K * 7 + N))
    w = nv.repack(gu.u8(packed), gu.u8(scales), float(d), N, K)
    rows = _sampled_rows(N, r)
    for M in (1, 2, 4, 8, 16):
        x_bits = synth.normal_bf16(r, (M, K))
        y = nv.gemm(gu.bits_to_bf16_tensor(x_bits), w)
        gu.check_device_status()
        yb = gu.tensor_to_bits(y)
        _, ref = dense.linear(x_bits, packed, scales, d, True, rows=rows)
        gu.compare(yb[:, rows], ref, f"M={M} K={K} N={N}")
        assert np.all(np.isfinite(formats.bf16_to_float(yb)))


@pytest.mark.parametrize("K,N", [(5120, 13824), (13824, 5120), (8192, 28672)])
def test_gemm_prefill_full_size_sampled(K, N):
    r = synth.rng(synth.seed_for(2, K + N))
    packed, scales, d = synth.weight_only(K, N, synth.seed_for(2, K * 7 + N))
    w = nv.repack(gu.u8(packed), gu.u8(scales), float(d), N, K)
    rows = _sampled_rows(N, r, n=24)
    for M, awq in ((512, False), (2048, True), (8192, False)):
        x_bits = synth.normal_bf16(r, (M, K))
        pqs = synth.awq_scale_bits(r, K) if awq else None
        y = nv.gemm(gu.bits_to_bf16_tensor(x_bits), w,
                    pre_quant_scale=gu.bits_to_bf16_tensor(pqs) if awq else None)
        gu.check_device_status()
        yb = gu.tensor_to_bits(y)
        _, ref = dense.linear(x_bits, packed, scales, d, True, pqs_bits=pqs, rows=rows)
        gu.compare(yb[:, rows], ref, f"M={M} K={K} N={N} awq={awq}")
        assert np.all(np.isfinite(formats.bf16_to_float(yb)))


@pytest.mark.parametrize("M,K,N", [(100, 1024, 20480), (300, 1040, 20480), (1000, 1024, 20480),
                                   (520, 4096, 2560), (777, 1536, 9990), (130, 2048, 19456)])
def test_gemm_tile_kernels_sampled(M, K, N):
    """Shapes that the tile planner sends to each dense tile kernel: the
    tensor-memory-A kernel with 128-token tiles (M=100) and 192-token tiles
    (partial last tile at M=300 and 130, K tail at K=1040, N tail at N=9990, a
    5-way K split at 520x4096x2560) and the shared-memory-operand kernel with
    256-token tiles (M=1000); every output row band of 16 is sampled."""
    r = synth.rng(synth.seed_for(6, M + K + N))
    packed, scales, d = synth.weight_only(K, N, synth.seed_for(6, M * 3 + K * 7 + N))
    w = nv.repack(gu.u8(packed), gu.u8(scales), float(d), N, K)
    rows = np.unique(np.concatenate([_sampled_rows(N, r, n=32), np.arange(0, N, 16), [N - 1]]))
    x_bits = synth.normal_bf16(r, (M, K))
    y = nv.gemm(gu.bits_to_bf16_tensor(x_bits), w)
    gu.check_device_status()
    yb = gu.tensor_to_bits(y)
    _, ref = dense.linear(x_bits, packed, scales, d, True, rows=rows)
    gu.compare(yb[:, rows], ref, f"tile M={M} K={K} N={N}")
    assert np.all(np.isfinite(formats.bf16_to_float(yb)))


@pytest.mark.parametrize("act", ["bf16", "f16"])
@pytest.mark.parametrize("M,K,N", [(100, 1024, 20480), (300, 1040, 20480), (1000, 1024, 20480), (520, 4096, 2560)])
def test_gemm_tile_kernels_awq(M, K, N, act):
    """The AWQ pre-quant scale on both tile kernels (x' = RN(x * s) by one pass
    before them): the tensor-memory-A kernel with 128- and 192-token tiles (K
    tail at K=1040), the shared-memory-operand kernel (M=1000) and a 5-way K
    split; BF16 and FP16; dropping the scale must fail the bar."""
    r = synth.rng(synth.seed_for(7, M + K + N) + (act == "f16"))
    packed, scales, d = synth.weight_only(K, N, synth.seed_for(7, M * 3 + K * 7 + N))
    w = nv.repack(gu.u8(packed), gu.u8(scales), float(d), N, K)
    rows = np.unique(np.concatenate([_sampled_rows(N, r, n=32), np.arange(0, N, 64), [N - 1]]))
    x_bits = synth.normal_act(r, (M, K), act)
    pqs = synth.awq_scale_bits(r, K, act)
    plan = nv.gemm_plan(M, N, K, has_pre_quant_scale=True)
    assert plan["kernel"] in ("tile_smem", "tile_tmem")
    assert plan["launches"] == (3 if plan["splits"] > 1 else 2)
    x = gu.bits_to_tensor(x_bits, act)
    y = nv.gemm(x, w, pre_quant_scale=gu.bits_to_tensor(pqs, act))
    gu.check_device_status()
    yb = gu.tensor_to_bits(y)
    _, ref = dense.linear(x_bits, packed, scales, d, True, pqs_bits=pqs, rows=rows, act=act)
    gu.compare(yb[:, rows], ref, f"tile AWQ M={M} K={K} N={N} {act}", act=act)
    plain = gu.tensor_to_bits(nv.gemm(x, w))
    with pytest.raises(AssertionError):
        gu.compare(plain[:, rows], ref, "tile dropped AWQ", act=act)


@pytest.mark.parametrize("M,K,N", [(64, 4096, 4096), (128, 14336, 4096), (256, 4096, 8192), (32, 4096, 4096)])
def test_gemm_mid_m_path_choice(M, K, N):
    """Between 17 and 511 tokens the path comes from a cost model (the
    streaming kernel expands the weights once per 16 tokens; the tile kernels
    once per tile, with a K split when the tiles alone leave SMs idle): these
    take the tile kernels with a K split, except M=32, which streams.  Sampled
    output rows against the oracle."""
    plan = nv.gemm_plan(M, N, K)
    assert plan["kernel"] == ("decode" if M == 32 else "tile_tmem" if M < 256 else plan["kernel"])
    r = synth.rng(synth.seed_for(8, M + K + N))
    packed, scales, d = synth.weight_only(K, N, synth.seed_for(8, M * 3 + K * 7 + N))
    w = nv.repack(gu.u8(packed), gu.u8(scales), float(d), N, K)
    rows = _sampled_rows(N, r, n=32)
    x_bits = synth.normal_bf16(r, (M, K))
    y = nv.gemm(gu.bits_to_bf16_tensor(x_bits), w)
    gu.check_device_status()
    yb = gu.tensor_to_bits(y)
    _, ref = dense.linear(x_bits, packed, scales, d, True, rows=rows)
    gu.compare(yb[:, rows], ref, f"mid M={M} K={K} N={N} ({plan['kernel']})")


def test_lm_head_full_size_sampled():
    K, N = 4096, 151936
    r = synth.rng(synth.seed_for(4, 0))
    packed, scales, d = synth.weight_only(K, N, synth.seed_for(4, 1))
    w = nv.repack(gu.u8(packed), gu.u8(scales), float(d), N, K)
    rows = _sampled_rows(N, r, n=64)
    for M in (1, 8, 256):
        x_bits = synth.normal_bf16(r, (M, K))
        y = nv.gemm(gu.bits_to_bf16_tensor(x_bits), w)
        gu.check_device_status()
        yb = gu.tensor_to_bits(y)
        _, ref = dense.linear(x_bits, packed, scales, d, True, rows=rows)
        gu.compare(yb[:, rows], ref, f"LM head M={M}")


@pytest.mark.parametrize("M,K,N", [(1000, 512, 8192), (600, 256, 1000)])
def test_gemm_tile_output_only_4_byte_aligned(M, K, N):
    """Y needs only 4-byte alignment: a tile GEMM into a view 4 bytes past an
    aligned buffer takes the element-wise stores and gives the same bits as
    into an aligned Y (the first shape plans the shared-memory tile kernel, the
    second a tile kernel with N % 8 == 0 but a ragged last column block)."""
    plan = nv.gemm_plan(M, N, K)
    assert plan["kernel"] in ("tile_smem", "tile_tmem")
    packed, scales, d = synth.weight_only(K, N, 31)
    w = nv.repack(gu.u8(packed), gu.u8(scales), float(d), N, K)
    x = gu.bits_to_bf16_tensor(synth.normal_bf16(synth.rng(32), (M, K)))
    y0 = nv.gemm(x, w)
    buf = torch.full((M * N + 2,), 7.0, dtype=torch.bfloat16, device="cuda")
    y1 = buf[2:].view(M, N)
    assert y1.data_ptr() % 16 == 4
    nv.gemm(x, w, out=y1)
    gu.check_device_status()
    assert np.array_equal(gu.tensor_to_bits(y0), gu.tensor_to_bits(y1))
    assert torch.all(buf[:2] == 7.0)


def test_gemm_bitwise_deterministic_across_runs():
    """Many waves of split-K clusters (ring reuse in every CTA): repeated runs must
    agree bit for bit -- the split-K reduction has a fixed order."""
    M, K, N = 64, 5120, 13824
    packed, scales, d = synth.weight_only(K, N, 11)
    w = nv.repack(gu.u8(packed), gu.u8(scales), float(d), N, K)
    x = gu.bits_to_bf16_tensor(synth.normal_bf16(synth.rng(5), (M, K)))
    outs = [gu.tensor_to_bits(nv.gemm(x, w)) for _ in range(5)]
    gu.check_device_status()
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


@pytest.mark.parametrize("K,N", [(720, 300), (2064, 1000), (64, 129), (4096, 512)])
def test_repack_from_swizzled_scales(K, N):
    """Scales given in the checkpoint's 128 x 4 swizzled layout repack to the same
    bytes as the linear view, and dequantize to the oracle's weights."""
    from tests.exact import swizzle_scales_by_tiles
    c = synth.gaussian_case(1, K, N, seed=300 + K + N)
    sw = swizzle_scales_by_tiles(c.scales, N, K)
    assert sw.size == nv.swizzled_scales_size(N, K) == formats.swizzled_scales_size(N, K)
    w_lin = gu.repack_case(c)
    w_swz = nv.repack(gu.u8(c.packed), gu.u8(sw), float(c.divisor), N, K, swizzled_scales=True)
    torch.cuda.synchronize()
    assert torch.equal(w_lin.buf, w_swz.buf)
    got = gu.tensor_to_bits(nv.dequant(w_swz))
    gu.check_device_status()
    want = dense.dequant(c.packed, formats.unswizzle_scales(sw, N, K), c.divisor, True, K)
    assert np.array_equal(got, want)
