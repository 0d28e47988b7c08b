"""The allocation-free MoE entry point against the regular one.

nvfp4_w4a16_moe_grouped_noalloc serves callers that cannot allocate device
memory (a plugin given no workspace by its host framework, code running while
allocation is not allowed): it runs the same layer on a fixed scratch array
inside the library.  This file is collected last so that a run stopping at the
first failure has already run every other test; it also passes on its own in
a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import w4a16_nvfp4_weight_gb300 as nv
from tests import gpu_util as gu
from w4a16_nvfp4_weight_gb300 import _lib, synth

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _experts(weights, N, K):
    size = nv.repack_size(N, K)
    buf = torch.empty(len(weights) * size, dtype=torch.uint8, device="cuda")
    for e, (p, s, d) in enumerate(weights):
        nv.repack(gu.u8(p), gu.u8(s), float(d), N, K, out=buf[e * size:(e + 1) * size])
    return buf


def _check_against_workspace_entry_point(lib, T, E, topk, H, I, seed):
    """Two allocation-free calls in a row give exactly the bytes of the regular
    entry point: both run the same kernels on the same inputs, only the memory
    that holds the intermediate tables and rows differs."""
    r = synth.rng(seed)
    fc1 = [synth.quantize(synth.normal_weight(r, 2 * I, H)) for _ in range(E)]
    fc2 = [synth.quantize(synth.normal_weight(r, H, I)) for _ in range(E)]
    c = synth.moe_case(T, seed + 1, E=E, topk=topk, H=H, I=I, weights=(fc1, fc2), awq=True)
    d1, d2 = _experts(fc1, 2 * I, H), _experts(fc2, H, I)
    x = gu.bits_to_bf16_tensor(c.x_bits)
    pqs = gu.bits_to_bf16_tensor(c.pqs_bits)
    logits = torch.from_numpy(np.ascontiguousarray(c.logits)).cuda()
    ref = gu.tensor_to_bits(nv.moe_grouped(x, logits, d1, d2, topk, I, fc1_pre_quant_scale=pqs))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert nv.moe_workspace_size(T, E, topk, H, I) <= lib.nvfp4_w4a16_moe_noalloc_scratch_bytes()
    for _ in range(2):                      # two calls in a row share the scratch array
        out = torch.full((T, H), 7.0, dtype=torch.bfloat16, device="cuda")
        idx = torch.empty((T, topk), dtype=torch.int32, device="cuda")
        st = lib.nvfp4_w4a16_moe_grouped_noalloc(_ptr(x), _ptr(logits), _ptr(d1), _ptr(d2), _ptr(pqs),
                                                 T, E, topk, H, I, _ptr(out), _ptr(idx), None, None, None,
                                                 stream)
        assert st == 0, lib.nvfp4_last_error().decode()
        gu.check_device_status()
        got = gu.tensor_to_bits(out)
        gu.compare(got, ref, "allocation-free MoE")
        assert np.array_equal(got, ref), "allocation-free MoE differs from the workspace entry point"


def test_noalloc_matches_workspace_entry_point(lib):
    # 48 tokens x top-4 over 16 experts: 12 rows per expert, the streaming kernels
    _check_against_workspace_entry_point(lib, 48, 16, 4, 256, 128, 2024)


def test_noalloc_tile_path_matches_workspace_entry_point(lib):
    # 128 tokens x top-4 over 16 experts: 32 rows per expert and I a multiple of
    # 128, so the layer gathers rows and runs the tcgen05 tile kernels, with the
    # gathered rows and FP32 partials at their own offsets in the scratch array
    _check_against_workspace_entry_point(lib, 128, 16, 4, 256, 128, 2026)


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    # 128 experts, top-8, hidden 2048, intermediate 768: 216 tokens need more than 16 MiB
    assert nv.moe_workspace_size(215, 128, 8, 2048, 768) <= lib.nvfp4_w4a16_moe_noalloc_scratch_bytes()
    assert nv.moe_workspace_size(216, 128, 8, 2048, 768) > lib.nvfp4_w4a16_moe_noalloc_scratch_bytes()
    st = lib.nvfp4_w4a16_moe_grouped_noalloc(None, None, None, None, None, 216, 128, 8, 2048, 768,
                                             None, None, None, None, None, None)
    assert st == 2
    assert "scratch" in lib.nvfp4_last_error().decode()
