"""The C-ABI library builds, loads, exports every function include/*.h
declares, and rejects bad arguments on the host before touching the GPU."""

import ctypes
import glob
import os
import re

import pytest

from w4a16_nvfp4_weight_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("nvfp4_repack", "nvfp4_dequant", "nvfp4_w4a16_gemm", "nvfp4_w4a16_moe_grouped",
              "nvfp4_repack_size", "nvfp4_last_error", "nvfp4_device_status",
              "nvfp4_dequant_f16", "nvfp4_w4a16_gemm_f16", "nvfp4_w4a16_moe_grouped_f16"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in sorted(_declared_functions()):
        assert hasattr(lib, n), f"{n} declared but not exported"
    assert set(_lib.SIGNATURES) == _declared_functions()
    assert lib.nvfp4_abi_version() == 2


def test_repack_size():
    lib = _lib.load(build_if_missing=True)
    assert lib.nvfp4_repack_size(0, 64) == 0
    assert lib.nvfp4_repack_size(4, 24) == 0                 # K % 16 != 0
    assert lib.nvfp4_repack_size(-1, 64) == 0
    # one 256-row tile, one 64-k block: header + two magnitude tables + 16 atoms
    assert lib.nvfp4_repack_size(1, 16) == 8448 + 16 * 576
    assert lib.nvfp4_repack_size(256, 64) == 8448 + 16 * 576
    assert lib.nvfp4_repack_size(257, 80) == 8448 + 2 * 2 * 16 * 576
    assert lib.nvfp4_repack_size(1000, 2064) % 256 == 0


def _err(lib):
    return lib.nvfp4_last_error().decode()


def test_gemm_rejects_bad_arguments_on_host(lib):
    V = ctypes.c_void_p
    good = V(0x10000)
    st = lib.nvfp4_w4a16_gemm(good, good, None, 4, 64, 24, good, None, 0, None)
    assert st == 2 and "multiple of 16" in _err(lib)
    st = lib.nvfp4_w4a16_gemm(good, good, None, -1, 64, 64, good, None, 0, None)
    assert st == 1
    st = lib.nvfp4_w4a16_gemm(None, good, None, 4, 64, 64, good, None, 0, None)
    assert st == 1 and "null" in _err(lib)
    st = lib.nvfp4_w4a16_gemm(V(0x10008), good, None, 4, 64, 64, good, None, 0, None)
    assert st == 3 and "X must be 16-byte aligned" in _err(lib)
    st = lib.nvfp4_w4a16_gemm(good, V(0x10010), None, 4, 64, 64, good, None, 0, None)
    assert st == 3 and "256-byte" in _err(lib)
    st = lib.nvfp4_w4a16_gemm(good, good, V(0x10002), 4, 64, 64, good, None, 0, None)
    assert st == 3 and "pre_quant_scale" in _err(lib)
    # zero rows / zero columns: OK, nothing launched (no device needed)
    assert lib.nvfp4_w4a16_gemm(None, None, None, 0, 64, 64, None, None, 0, None) == 0
    assert lib.nvfp4_w4a16_gemm(None, None, None, 4, 0, 64, None, None, 0, None) == 0


def test_repack_and_dequant_reject_bad_arguments_on_host(lib):
    V = ctypes.c_void_p
    good = V(0x10000)
    assert lib.nvfp4_repack(good, good, 448.0, 1, 16, 40, good, 1 << 20, None) == 2
    assert lib.nvfp4_repack(None, good, 448.0, 1, 16, 64, good, 1 << 20, None) == 1
    assert lib.nvfp4_repack(good, good, 448.0, 2, 16, 64, good, 1 << 20, None) == 1
    assert lib.nvfp4_repack(good, good, 448.0, 1, 16, 64, V(0x10080), 1 << 20, None) == 3
    assert lib.nvfp4_repack(good, good, 448.0, 1, 16, 64, good, 100, None) == 4
    assert "needs" in _err(lib)
    assert lib.nvfp4_repack(good, good, 0.0, 0, 16, 64, good, 1 << 20, None) == 1
    assert lib.nvfp4_repack(good, good, 0.0, 1, 16, 64, good, 1 << 20, None) == 1   # 1/0
    assert lib.nvfp4_repack(good, good, float("nan"), 1, 16, 64, good, 1 << 20, None) == 1
    assert lib.nvfp4_dequant(good, 16, 40, good, None) == 2
    assert lib.nvfp4_dequant(V(0x10010), 16, 64, good, None) == 3
    assert lib.nvfp4_dequant(good, 16, 64, V(0x10004), None) == 3


def test_python_binding_refuses_non_bf16_activations():
    import torch
    import w4a16_nvfp4_weight_gb300 as nv
    w = nv.NVFP4Weight(torch.empty(16, dtype=torch.uint8), 16, 64)
    with pytest.raises(nv.Nvfp4Error):
        nv.gemm(torch.zeros(2, 64, dtype=torch.float8_e4m3fn), w)
    with pytest.raises(nv.Nvfp4Error):
        nv.gemm(torch.zeros(2, 64, dtype=torch.bfloat16), w)     # CPU tensor


def test_swizzled_scales_size_and_layout_flag(lib):
    assert lib.nvfp4_swizzled_scales_size(1, 16) == 128 * 4
    assert lib.nvfp4_swizzled_scales_size(129, 80) == 256 * 8
    assert lib.nvfp4_swizzled_scales_size(0, 16) == 0
    V = ctypes.c_void_p
    good = V(0x10000)
    st = lib.nvfp4_repack_ex(good, good, 7, 1.0, 1, 16, 64, good, 1 << 20, None)
    assert st == 1 and "scale_layout" in _err(lib)


def test_moe_and_mlp_reject_bad_arguments_on_host(lib):
    """MoE, dense-MLP and AWQ-finalization entry points validate before any
    launch (status 1 invalid argument, 2 unsupported shape, 3 alignment,
    4 workspace); T = 0 returns OK without touching a pointer."""
    V = ctypes.c_void_p
    g, big = V(0x100000), 1 << 40

    def moe(X=g, lg=g, w1=g, w2=g, pqs=None, T=1, E=128, k=8, H=2048, I=768, act=0, split=0, f16=0,
            out=g, ws=g, wsb=big):
        return lib.nvfp4_w4a16_moe_grouped_ex(X, lg, w1, w2, pqs, T, E, k, H, I, act, split, f16,
                                              out, None, None, None, None, ws, wsb, None)

    assert moe(f16=2) == 1
    assert moe(act=3) == 1 and "SWIGLU" in _err(lib)
    assert moe(act=1, split=1) == 1                       # shards only with the gated experts
    assert moe(T=-1) == 1
    assert moe(E=0) == 2 and moe(E=257) == 2
    assert moe(k=0) == 2 and moe(E=4, k=5) == 2 and moe(k=17) == 2
    assert moe(H=100) == 2 and moe(I=0) == 2
    assert moe(X=None, lg=None, w1=None, w2=None, out=None, ws=None, wsb=0, T=0) == 0
    assert moe(X=None) == 1 and "null" in _err(lib)
    assert moe(X=V(0x100008)) == 3
    assert moe(lg=V(0x100002)) == 3
    assert moe(w1=V(0x100010)) == 3
    assert moe(pqs=V(0x100008)) == 3
    assert moe(wsb=0) == 4 and "needs" in _err(lib)
    assert moe(ws=V(0x100040)) == 3
    assert moe(T=10_000_000) == 2                         # more work items than one grid dimension holds

    def route(lg=g, T=4, E=128, k=8, idx=g, p=g, perm=g, inv=g, offs=g):
        return lib.nvfp4_moe_route(lg, T, E, k, idx, p, perm, inv, offs, None)

    assert route(T=-1) == 1
    assert route(E=0) == 2 and route(E=257) == 2 and route(E=4, k=5) == 2 and route(k=17) == 2
    assert route(T=1 << 28) == 2                          # T * topk past int32 slot indices
    assert route(lg=None, idx=None, p=None, perm=None, inv=None, offs=None, T=0) == 0
    assert route(inv=None) == 1 and "null" in _err(lib)
    assert route(perm=V(0x100002)) == 3

    def mlp(X=g, w1=g, w2=g, pqs=None, T=4, H=4096, I=14336, out=g, ws=g, wsb=big):
        return lib.nvfp4_w4a16_mlp(X, w1, w2, pqs, T, H, I, out, ws, wsb, None)

    assert mlp(T=-1) == 1
    assert mlp(H=100) == 2 and mlp(I=0) == 2
    assert mlp(X=None, w1=None, w2=None, out=None, ws=None, wsb=0, T=0) == 0
    assert mlp(w2=None) == 1
    assert mlp(out=V(0x100008)) == 3
    assert mlp(w1=V(0x100080)) == 3
    assert mlp(pqs=V(0x100004)) == 3
    assert mlp(wsb=16) == 4
    assert mlp(ws=V(0x100010)) == 3
    assert lib.nvfp4_w4a16_mlp_workspace(4, 4096, 14336) > lib.nvfp4_w4a16_mlp_workspace(1, 4096, 14336) > 0

    fin = lib.nvfp4_moe_finalize_pre_quant_scale
    assert fin(g, g, 0, 64, 0, g, None) == 1
    assert fin(g, g, 2, 0, 0, g, None) == 1
    assert fin(g, g, 2, 64, 2, g, None) == 1
    assert fin(None, g, 2, 64, 0, g, None) == 1
    assert fin(g, g, 2, 64, 0, V(0x100001), None) == 3


def test_gemm_plan_on_host(lib):
    """The launch plan query: host only, the same shape rules the GEMM entry
    points use (without a device 148 SMs are assumed; with one, its SM count
    decides the wave sizes, so the exact tile plans are checked only at the SM
    counts they were derived for)."""
    import torch

    import w4a16_nvfp4_weight_gb300 as nv

    assert nv.gemm_plan(0, 4096, 4096) == {"kernel": "none", "tokens": 0, "splits": 0, "launches": 0}
    for M in (1, 8, 9, 16):
        p = nv.gemm_plan(M, 4096, 4096)
        assert p["kernel"] == "decode" and p["tokens"] == (8 if M <= 8 else 16) and p["launches"] == 1
        assert 1 <= p["splits"] <= 8
        # the decode kernel applies the AWQ scale itself: no extra pass, no workspace
        assert nv.gemm_plan(M, 4096, 4096, has_pre_quant_scale=True)["launches"] == 1
        assert nv.gemm_workspace_size(M, 4096, 4096, True) == 0
    # few output tiles below M = 512 stay on the streaming kernel
    assert nv.gemm_plan(300, 1000, 2064)["kernel"] == "decode"
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 148
    if sms in (148, 152):
        # (M, N, K): tensor-memory-A tiles (220 tiles of 216 blocks: a 2-way K split
        # plus its reduction pass fills the waves better), shared-memory tiles, and
        # a K split with its reduction pass
        assert nv.gemm_plan(2048, 5120, 13824) == {"kernel": "tile_tmem", "tokens": 192, "splits": 2, "launches": 2}
        assert nv.gemm_plan(2048, 13824, 5120) == {"kernel": "tile_smem", "tokens": 256, "splits": 1, "launches": 1}
        # the tile kernels take the AWQ-scaled activations from one pass before
        # them (its buffer in the workspace); the K split adds its reduction pass
        p = nv.gemm_plan(512, 5120, 13824, has_pre_quant_scale=True)
        assert p["kernel"] == "tile_smem" and p["splits"] > 1 and p["launches"] == 3
        assert nv.gemm_workspace_size(512, 5120, 13824, True) == \
            nv.gemm_workspace_size(512, 5120, 13824, False) + 512 * 13824 * 2

    out = [ctypes.c_int(0) for _ in range(4)]
    refs = [ctypes.byref(o) for o in out]
    assert lib.nvfp4_w4a16_gemm_plan(4, 64, 24, 0, *refs) == 2
    assert lib.nvfp4_w4a16_gemm_plan(-1, 64, 64, 0, *refs) == 1
    assert lib.nvfp4_w4a16_gemm_plan(4, 64, 64, 2, *refs) == 1
    assert lib.nvfp4_w4a16_gemm_plan(4, 64, 64, 0, None, *refs[1:]) == 1


def test_moe_plan_on_host(lib):
    """The MoE path query: host only, the choice the layer makes from the
    average routed rows per expert and the expected units per SM (the config
    layer E=128, top-8, H=2048, I=768 at T = 1, 16, 256, 4096)."""
    import w4a16_nvfp4_weight_gb300 as nv

    E, k, H, I = 128, 8, 2048, 768
    assert nv.moe_plan(0, E, k, H, I) == {"path": "none", "rows_per_item": 0}
    assert nv.moe_plan(1, E, k, H, I) == {"path": "single_token", "rows_per_item": 8}
    assert nv.moe_plan(2, E, k, H, I) == {"path": "stream_split", "rows_per_item": 8}
    assert nv.moe_plan(1, 32, 16, H, I)["path"] == "stream_split"      # top-16: beyond one portable cluster
    assert nv.moe_plan(16, E, k, H, I) == {"path": "stream_persistent", "rows_per_item": 8}
    assert nv.moe_plan(256, E, k, H, I) == {"path": "stream_persistent", "rows_per_item": 32}
    assert nv.moe_plan(160, E, k, H, I) == {"path": "stream_persistent", "rows_per_item": 16}
    assert nv.moe_plan(4096, E, k, H, I) == {"path": "tile", "rows_per_item": 256}
    # non-gated experts have half the FC1 column groups
    assert nv.moe_plan(16, E, k, H, I, "relu2")["path"] in ("stream_split", "stream_persistent")

    path, rows = ctypes.c_int(0), ctypes.c_int(0)
    refs = [ctypes.byref(path), ctypes.byref(rows)]
    assert lib.nvfp4_w4a16_moe_plan(4, 8, 2, 64, 64, 0, *refs) == 0 and path.value == 1
    assert lib.nvfp4_w4a16_moe_plan(1, 8, 2, 64, 64, 0, *refs) == 0 and path.value == 4
    assert lib.nvfp4_w4a16_moe_plan(-1, 8, 2, 64, 64, 0, *refs) == 1
    assert lib.nvfp4_w4a16_moe_plan(4, 8, 2, 64, 64, 3, *refs) == 1
    assert lib.nvfp4_w4a16_moe_plan(4, 0, 2, 64, 64, 0, *refs) == 2
    assert lib.nvfp4_w4a16_moe_plan(4, 8, 9, 64, 64, 0, *refs) == 2
    assert lib.nvfp4_w4a16_moe_plan(4, 8, 2, 96, 64, 0, *refs) == 2
    assert lib.nvfp4_w4a16_moe_plan(4, 8, 2, 64, 64, 0, None, refs[1]) == 1
