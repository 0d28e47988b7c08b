"""W4A16 NVFP4 weight-only GEMM for GB300 (sm_103a).

Thin Python binding over the C ABI in ``include/nvfp4_w4a16.h``: it allocates
outputs with torch, passes raw device pointers and the current CUDA stream, and
turns non-OK statuses into ``Nvfp4Error``.  Every step of the computation runs
in the library's CUDA kernels; there is no Python or CPU fallback.

    w = repack(packed_u8, scales_u8, divisor, N, K, global_is_divisor=True)
    y = gemm(x_bf16, w)                       # [M, K] -> [M, N]
    y = gemm(x_bf16, w, pre_quant_scale=s)    # AWQ checkpoints
    y = gemm(x_fp16, w)                       # FP16 activations: FP16 weights and output

The activation dtype (torch.bfloat16 or torch.float16) selects the entry
point (nvfp4_w4a16_gemm or nvfp4_w4a16_gemm_f16, and likewise for the MoE
layer and the dequant).
"""

import ctypes

import torch

from . import _lib
from ._lib import Nvfp4Error

__all__ = ["Nvfp4Error", "NVFP4Weight", "repack", "repack_size", "swizzled_scales_size", "dequant", "gemm",
           "gemm_workspace_size", "gemm_plan", "moe_grouped", "moe_plan", "moe_route", "moe_workspace_size",
           "moe_finalize_pre_quant_scale",
           "mlp", "mlp_workspace_size",
           "device_status",
           "abi_version"]


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


_ACT_DTYPES = (torch.bfloat16, torch.float16)


def _act_dtype(x, name):
    if not isinstance(x, torch.Tensor) or x.dtype not in _ACT_DTYPES:
        raise Nvfp4Error(1, f"{name} must be a torch.bfloat16 or torch.float16 CUDA tensor")
    return x.dtype


def _require_cuda(t, name, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise Nvfp4Error(1, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise Nvfp4Error(1, f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise Nvfp4Error(1, f"{name} must be {dtype}, got {t.dtype}")


def abi_version():
    return _lib.load().nvfp4_abi_version()


def repack_size(N, K):
    return int(_lib.load().nvfp4_repack_size(N, K))


class NVFP4Weight:
    """A repacked NVFP4 weight (device buffer) with its logical shape [N, K]."""

    def __init__(self, buf, N, K):
        self.buf, self.N, self.K = buf, int(N), int(K)

    @property
    def nbytes(self):
        return self.buf.numel()


def repack(packed, scales, global_scale, N, K, global_is_divisor=True, out=None, swizzled_scales=False):
    """Checkpoint tensors (uint8 [N, K/2] codes, uint8 E4M3 scales) -> NVFP4Weight.
    ``scales`` is the linear [N, K/16] view, or with ``swizzled_scales`` the
    checkpoint's 128 x 4 swizzled layout (swizzled_scales_size(N, K) bytes).
    ``global_scale`` is a Python float (the stored value)."""
    h = _lib.load()
    _require_cuda(packed, "packed", torch.uint8)
    _require_cuda(scales, "scales", torch.uint8)
    size = int(h.nvfp4_repack_size(N, K))
    if out is None:
        out = torch.empty(max(size, 256), dtype=torch.uint8, device=packed.device)
    if swizzled_scales:
        if scales.numel() < swizzled_scales_size(N, K):
            raise Nvfp4Error(2, f"swizzled scales need {swizzled_scales_size(N, K)} bytes")
        _lib.check(h.nvfp4_repack_ex(_ptr(packed), _ptr(scales), 1, float(global_scale),
                                     1 if global_is_divisor else 0, N, K, _ptr(out), out.numel(), _stream()))
    else:
        _lib.check(h.nvfp4_repack(_ptr(packed), _ptr(scales), float(global_scale),
                                  1 if global_is_divisor else 0, N, K, _ptr(out), out.numel(), _stream()))
    return NVFP4Weight(out, N, K)


def swizzled_scales_size(N, K):
    return int(_lib.load().nvfp4_swizzled_scales_size(N, K))


def dequant(w, out=None, dtype=torch.bfloat16):
    """[N, K] weight exactly as the GEMM kernels see it, in ``dtype`` (the
    activation type: torch.bfloat16 or torch.float16)."""
    h = _lib.load()
    if dtype not in _ACT_DTYPES:
        raise Nvfp4Error(1, "dtype must be torch.bfloat16 or torch.float16")
    if out is None:
        out = torch.empty((w.N, w.K), dtype=dtype, device=w.buf.device)
    _require_cuda(out, "out", dtype)
    fn = h.nvfp4_dequant_f16 if dtype == torch.float16 else h.nvfp4_dequant
    _lib.check(fn(_ptr(w.buf), w.N, w.K, _ptr(out), _stream()))
    return out


def gemm_workspace_size(M, N, K, has_pre_quant_scale=False):
    return int(_lib.load().nvfp4_w4a16_gemm_workspace(M, N, K, 1 if has_pre_quant_scale else 0))


GEMM_KERNELS = {-1: "none", 0: "decode", 1: "tile_smem", 2: "tile_tmem"}


def gemm_plan(M, N, K, has_pre_quant_scale=False):
    """The launch plan of gemm() for an M x N x K problem on the current device:
    dict(kernel=name, tokens=rows per CTA tile, splits=K splits,
    launches=kernels per call).  Host only."""
    h = _lib.load()
    out = [ctypes.c_int(0) for _ in range(4)]
    _lib.check(h.nvfp4_w4a16_gemm_plan(M, N, K, 1 if has_pre_quant_scale else 0,
                                       *[ctypes.byref(o) for o in out]))
    kernel, tokens, splits, launches = (o.value for o in out)
    return {"kernel": GEMM_KERNELS[kernel], "tokens": tokens, "splits": splits, "launches": launches}


def gemm(x, w, pre_quant_scale=None, out=None, workspace=None):
    """Y[M, N] = X'[M, K] . W^T in the activation type of x (BF16 or FP16),
    X' = X or RN(X * pre_quant_scale)."""
    h = _lib.load()
    dt = _act_dtype(x, "x")
    _require_cuda(x, "x", dt)
    if x.dim() != 2 or x.shape[1] != w.K:
        raise Nvfp4Error(2, f"x must be [M, {w.K}], got {tuple(x.shape)}")
    if pre_quant_scale is not None:
        _require_cuda(pre_quant_scale, "pre_quant_scale", dt)
        if pre_quant_scale.numel() != w.K:
            raise Nvfp4Error(2, f"pre_quant_scale must have {w.K} elements")
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, w.N), dtype=dt, device=x.device)
    _require_cuda(out, "out", dt)
    need = gemm_workspace_size(M, w.N, w.K, pre_quant_scale is not None)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_bytes = workspace.numel() if workspace is not None else 0
    fn = h.nvfp4_w4a16_gemm_f16 if dt == torch.float16 else h.nvfp4_w4a16_gemm
    _lib.check(fn(_ptr(x), _ptr(w.buf), _ptr(pre_quant_scale), M, w.N, w.K,
                  _ptr(out), _ptr(workspace), ws_bytes, _stream()))
    return out


def moe_route(router_logits, topk):
    """The MoE routing step alone: dict(idx [T, topk] int32, p [T, topk]
    float32, perm [T*topk] int32, inv [T*topk] int32, offsets [E+1] int32)."""
    h = _lib.load()
    _require_cuda(router_logits, "router_logits", torch.float32)
    if router_logits.dim() != 2:
        raise Nvfp4Error(2, f"router_logits must be [T, E], got {tuple(router_logits.shape)}")
    T, E = router_logits.shape
    dev = router_logits.device
    idx = torch.empty((T, topk), dtype=torch.int32, device=dev)
    p = torch.empty((T, topk), dtype=torch.float32, device=dev)
    perm = torch.empty(T * topk, dtype=torch.int32, device=dev)
    inv = torch.empty(T * topk, dtype=torch.int32, device=dev)
    offsets = torch.zeros(E + 1, dtype=torch.int32, device=dev)
    _lib.check(h.nvfp4_moe_route(_ptr(router_logits), T, E, topk, _ptr(idx), _ptr(p), _ptr(perm), _ptr(inv),
                                 _ptr(offsets), _stream()))
    return dict(idx=idx, p=p, perm=perm, inv=inv, offsets=offsets)


def moe_workspace_size(T, E, topk, H, I):
    return int(_lib.load().nvfp4_w4a16_moe_workspace(T, E, topk, H, I))


MOE_ACTIVATIONS = {"swiglu": 0, "relu2": 1, "silu": 2}
MOE_PATHS = {0: "none", 1: "stream_split", 2: "stream_persistent", 3: "tile", 4: "single_token"}


def moe_plan(T, E, topk, H, I, activation="swiglu"):
    """The kernels moe_grouped() would run on the current device: dict(path=
    "single_token" | "stream_split" | "stream_persistent" | "tile" | "none",
    rows_per_item).
    Host only."""
    if activation not in MOE_ACTIVATIONS:
        raise Nvfp4Error(1, f"activation must be one of {sorted(MOE_ACTIVATIONS)}")
    h = _lib.load()
    path, rows = ctypes.c_int(0), ctypes.c_int(0)
    _lib.check(h.nvfp4_w4a16_moe_plan(T, E, topk, H, I, MOE_ACTIVATIONS[activation],
                                      ctypes.byref(path), ctypes.byref(rows)))
    return {"path": MOE_PATHS[path.value], "rows_per_item": rows.value}


def moe_grouped(x, router_logits, fc1, fc2, topk, I, fc1_pre_quant_scale=None, out=None,
                return_routing=False, workspace=None, activation="swiglu", fc1_split=False):
    """Top-k MoE layer.  ``fc1``/``fc2``: uint8 device buffers holding E repacked
    expert weights back to back ([2I, H] and [H, I] each).  x is BF16 or FP16;
    out and fc1_pre_quant_scale have its type.  ``activation`` "relu2" or
    "silu": non-gated experts, fc1 holds E repacked [I, H] weights.
    ``fc1_split``: gated experts whose gate and up projections are repacked
    separately (each with its own global), gate then up per expert."""
    h = _lib.load()
    dt = _act_dtype(x, "x")
    _require_cuda(x, "x", dt)
    _require_cuda(router_logits, "router_logits", torch.float32)
    if fc1_pre_quant_scale is not None:
        _require_cuda(fc1_pre_quant_scale, "fc1_pre_quant_scale", dt)
    T, H = x.shape
    E = router_logits.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=dt, device=x.device)
    _require_cuda(out, "out", dt)
    dev = x.device
    idx = wts = perm = offs = None
    if return_routing:
        idx = torch.empty((T, topk), dtype=torch.int32, device=dev)
        wts = torch.empty((T, topk), dtype=torch.float32, device=dev)
        perm = torch.empty(T * topk, dtype=torch.int32, device=dev)
        offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    need = moe_workspace_size(T, E, topk, H, I)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() if workspace is not None else 0
    if activation not in MOE_ACTIVATIONS:
        raise Nvfp4Error(1, f"activation must be one of {sorted(MOE_ACTIVATIONS)}")
    if activation != "swiglu" or fc1_split:
        _lib.check(h.nvfp4_w4a16_moe_grouped_ex(
            _ptr(x), _ptr(router_logits), _ptr(fc1), _ptr(fc2), _ptr(fc1_pre_quant_scale),
            T, E, topk, H, I, MOE_ACTIVATIONS[activation], 1 if fc1_split else 0,
            1 if dt == torch.float16 else 0, _ptr(out), _ptr(idx), _ptr(wts), _ptr(perm), _ptr(offs),
            _ptr(workspace), ws_bytes, _stream()))
    else:
        fn = h.nvfp4_w4a16_moe_grouped_f16 if dt == torch.float16 else h.nvfp4_w4a16_moe_grouped
        _lib.check(fn(
            _ptr(x), _ptr(router_logits), _ptr(fc1), _ptr(fc2), _ptr(fc1_pre_quant_scale),
            T, E, topk, H, I, _ptr(out), _ptr(idx), _ptr(wts), _ptr(perm), _ptr(offs),
            _ptr(workspace), ws_bytes, _stream()))
    if return_routing:
        return out, dict(idx=idx, p=wts, perm=perm, offsets=offs)
    return out


def moe_finalize_pre_quant_scale(w1_pre_quant_scale, w3_pre_quant_scale, out=None):
    """[H] FC1 activation scale = max over experts of max(w3_e, w1_e); inputs [E, H]
    BF16 or FP16 (same type), the output has their type."""
    h = _lib.load()
    dt = _act_dtype(w1_pre_quant_scale, "w1_pre_quant_scale")
    _require_cuda(w1_pre_quant_scale, "w1_pre_quant_scale", dt)
    _require_cuda(w3_pre_quant_scale, "w3_pre_quant_scale", dt)
    if w1_pre_quant_scale.shape != w3_pre_quant_scale.shape or w1_pre_quant_scale.dim() != 2:
        raise Nvfp4Error(2, "w1/w3 pre-quant scales must both be [E, H]")
    E, H = w1_pre_quant_scale.shape
    if out is None:
        out = torch.empty(H, dtype=dt, device=w1_pre_quant_scale.device)
    _lib.check(h.nvfp4_moe_finalize_pre_quant_scale(_ptr(w1_pre_quant_scale), _ptr(w3_pre_quant_scale), E, H,
                                                    1 if dt == torch.float16 else 0, _ptr(out), _stream()))
    return out


def mlp_workspace_size(T, H, I):
    return int(_lib.load().nvfp4_w4a16_mlp_workspace(T, H, I))


def mlp(x, fc1, fc2, fc1_pre_quant_scale=None, out=None, workspace=None):
    """Dense gated MLP: out = FC2(RN(silu(g) * u)), [g; u] = FC1(x').
    ``fc1``: NVFP4Weight [2I, H] (gate rows then up rows), ``fc2``: NVFP4Weight
    [H, I]; x is BF16 or FP16 [T, H] and out has its type."""
    h = _lib.load()
    dt = _act_dtype(x, "x")
    _require_cuda(x, "x", dt)
    T, H = x.shape
    I = fc1.N // 2
    if fc1.K != H or fc1.N != 2 * I or fc2.N != H or fc2.K != I:
        raise Nvfp4Error(2, f"fc1 must be [2I, {H}] and fc2 [{H}, I]; got {fc1.N}x{fc1.K} and {fc2.N}x{fc2.K}")
    if fc1_pre_quant_scale is not None:
        _require_cuda(fc1_pre_quant_scale, "fc1_pre_quant_scale", dt)
    if out is None:
        out = torch.empty((T, H), dtype=dt, device=x.device)
    _require_cuda(out, "out", dt)
    need = mlp_workspace_size(T, H, I)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_bytes = workspace.numel() if workspace is not None else 0
    fn = h.nvfp4_w4a16_mlp_f16 if dt == torch.float16 else h.nvfp4_w4a16_mlp
    _lib.check(fn(_ptr(x), _ptr(fc1.buf), _ptr(fc2.buf), _ptr(fc1_pre_quant_scale), T, H, I,
                  _ptr(out), _ptr(workspace), ws_bytes, _stream()))
    return out


def device_status(clear=True):
    """Synchronize the current stream and return (and clear) the device status word."""
    h = _lib.load()
    v = ctypes.c_int(0)
    _lib.check(h.nvfp4_device_status(ctypes.byref(v), 1 if clear else 0, _stream()))
    return v.value
