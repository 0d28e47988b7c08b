"""ctypes handle on the C ABI declared in include/nvfp4_w4a16.h.

Loading fails loudly when the library has not been built: there is no other
implementation to fall back to.
"""

import ctypes
import os

from . import build_lib

c_i64 = ctypes.c_int64
c_int = ctypes.c_int
c_size = ctypes.c_size_t
c_vp = ctypes.c_void_p
c_float = ctypes.c_float

# name -> (restype, argtypes), mirroring include/nvfp4_w4a16.h
SIGNATURES = {
    "nvfp4_abi_version": (c_int, []),
    "nvfp4_last_error": (ctypes.c_char_p, []),
    "nvfp4_device_status": (c_int, [ctypes.POINTER(c_int), c_int, c_vp]),
    "nvfp4_repack_size": (c_size, [c_i64, c_i64]),
    "nvfp4_repack": (c_int, [c_vp, c_vp, c_float, c_int, c_i64, c_i64, c_vp, c_size, c_vp]),
    "nvfp4_swizzled_scales_size": (c_size, [c_i64, c_i64]),
    "nvfp4_repack_ex": (c_int, [c_vp, c_vp, c_int, c_float, c_int, c_i64, c_i64, c_vp, c_size, c_vp]),
    "nvfp4_dequant": (c_int, [c_vp, c_i64, c_i64, c_vp, c_vp]),
    "nvfp4_dequant_f16": (c_int, [c_vp, c_i64, c_i64, c_vp, c_vp]),
    "nvfp4_w4a16_gemm_workspace": (c_size, [c_i64, c_i64, c_i64, c_int]),
    "nvfp4_w4a16_gemm": (c_int, [c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_size, c_vp]),
    "nvfp4_w4a16_gemm_f16": (c_int, [c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_size, c_vp]),
    "nvfp4_w4a16_gemm_plan": (c_int, [c_i64, c_i64, c_i64, c_int, c_vp, c_vp, c_vp, c_vp]),
    "nvfp4_w4a16_moe_plan": (c_int, [c_i64, c_int, c_int, c_i64, c_i64, c_int, c_vp, c_vp]),
    "nvfp4_moe_route": (c_int, [c_vp, c_i64, c_int, c_int, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "nvfp4_w4a16_moe_workspace": (c_size, [c_i64, c_int, c_int, c_i64, c_i64]),
    "nvfp4_w4a16_moe_grouped": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_int, c_int, c_i64,
                                        c_i64, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_size, c_vp]),
    "nvfp4_w4a16_moe_grouped_f16": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_int, c_int, c_i64,
                                            c_i64, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_size, c_vp]),
    "nvfp4_w4a16_moe_grouped_ex": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_int, c_int, c_i64,
                                           c_i64, c_int, c_int, c_int, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                           c_size, c_vp]),
    "nvfp4_moe_finalize_pre_quant_scale": (c_int, [c_vp, c_vp, c_int, c_i64, c_int, c_vp, c_vp]),
    "nvfp4_w4a16_mlp_workspace": (c_size, [c_i64, c_i64, c_i64]),
    "nvfp4_w4a16_mlp": (c_int, [c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_size, c_vp]),
    "nvfp4_w4a16_mlp_f16": (c_int, [c_vp, c_vp, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_size, c_vp]),
    "nvfp4_w4a16_moe_noalloc_scratch_bytes": (c_size, []),
    "nvfp4_w4a16_moe_grouped_noalloc": (c_int, [c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_int, c_int, c_i64,
                                                c_i64, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
}

STATUS_NAMES = {
    0: "NVFP4_OK", 1: "NVFP4_ERR_INVALID_ARG", 2: "NVFP4_ERR_UNSUPPORTED_SHAPE",
    3: "NVFP4_ERR_ALIGNMENT", 4: "NVFP4_ERR_WORKSPACE", 5: "NVFP4_ERR_CUDA",
    6: "NVFP4_ERR_TIMEOUT", 7: "NVFP4_ERR_BAD_WEIGHT",
}


class Nvfp4Error(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_handle = None


def path():
    return build_lib.LIB


def load(build_if_missing=False):
    """Load the shared library (optionally building it first)."""
    global _handle
    if _handle is not None:
        return _handle
    if build_if_missing:
        build_lib.build()
    if not os.path.exists(build_lib.LIB):
        raise RuntimeError(
            f"CUDA library not built ({build_lib.LIB} missing); run "
            "`python -c 'import __graft_entry__ as g; g.build()'` first")
    h = ctypes.CDLL(build_lib.LIB)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(h, name)
        fn.restype = res
        fn.argtypes = args
    _handle = h
    return h


def check(status):
    if status != 0:
        msg = load().nvfp4_last_error().decode(errors="replace")
        raise Nvfp4Error(status, msg)
