"""ctypes view of the C ABI declared in include/moe.h (structs and symbols).

Loading fails loudly when libmoe.so has not been built: there is no other
implementation of the layer to fall back to.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB

c_i32 = ctypes.c_int32
c_vp = ctypes.c_void_p
c_fp = ctypes.POINTER(ctypes.c_float)
c_ip = ctypes.POINTER(ctypes.c_int32)


class MoeDesc(ctypes.Structure):
    _fields_ = [("n_tok", c_i32), ("d_model", c_i32), ("d_ff", c_i32), ("n_exp", c_i32), ("top_k", c_i32),
                ("gate", c_i32), ("use_bias", c_i32), ("n_shared", c_i32), ("d_ff_shared", c_i32),
                ("precision", c_i32)]


class MoeExpertWeights(ctypes.Structure):
    _fields_ = [("w1", c_vp), ("w3", c_vp), ("w2", c_vp), ("ws1", c_vp), ("ws3", c_vp), ("ws2", c_vp)]


class MoeFfnSaved(ctypes.Structure):
    _fields_ = [("a1", c_vp), ("a3", c_vp), ("h", c_vp), ("a1s", c_vp), ("a3s", c_vp), ("hs", c_vp)]


class MoeFwdState(ctypes.Structure):
    _fields_ = [("x", c_vp), ("x_perm", c_vp), ("logits", c_vp), ("topk_idx", c_vp), ("topk_w", c_vp),
                ("offsets", c_vp), ("row_of_copy", c_vp), ("copy_of_row", c_vp), ("a1", c_vp), ("a3", c_vp),
                ("h", c_vp), ("y_perm", c_vp), ("a1s", c_vp), ("a3s", c_vp), ("hs", c_vp),
                ("offsets_full", c_vp), ("copy_of_row_full", c_vp)]


class MoeGrads(ctypes.Structure):
    _fields_ = [("dx", c_vp), ("dw_gate", c_vp), ("dw1", c_vp), ("dw3", c_vp), ("dw2", c_vp), ("dws1", c_vp),
                ("dws3", c_vp), ("dws2", c_vp), ("dg", c_vp), ("dlogits", c_vp)]


class MoeExpertWeightsMx(ctypes.Structure):
    _fields_ = [(n, c_vp) for n in ("w1", "w1_scale", "w3", "w3_scale", "w2", "w2_scale",
                                    "ws1", "ws1_scale", "ws3", "ws3_scale", "ws2", "ws2_scale")]


# name -> (restype, argtypes); every entry point of include/moe.h
SIGNATURES = {
    "moe_abi_version": (c_i32, []),
    "moe_status_string": (ctypes.c_char_p, [c_i32]),
    "moe_workspace_size": (c_i32, [ctypes.POINTER(MoeDesc), ctypes.POINTER(ctypes.c_size_t),
                                   ctypes.POINTER(ctypes.c_size_t)]),
    "moe_workspace_init": (c_i32, [c_vp, ctypes.c_size_t, c_vp]),
    "moe_get_device_status": (c_i32, [c_vp, c_ip, c_vp]),
    "moe_route": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                          ctypes.c_size_t, c_vp]),
    "moe_route_from_logits": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                      ctypes.c_size_t, c_vp]),
    "moe_route_permute": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                  c_vp, c_vp, c_vp, ctypes.c_size_t, c_vp]),
    "moe_permute": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, ctypes.c_size_t,
                            c_vp]),
    "moe_grouped_ffn": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, c_vp, c_vp, ctypes.POINTER(MoeExpertWeights),
                                ctypes.POINTER(MoeFfnSaved), c_vp, c_vp, c_vp, ctypes.c_size_t, c_vp]),
    "moe_combine": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "moe_backward": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, ctypes.POINTER(MoeExpertWeights),
                             ctypes.POINTER(MoeFwdState), c_vp, ctypes.POINTER(MoeGrads), c_vp, ctypes.c_size_t,
                             c_vp]),
    "moe_update_bias": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, c_vp, ctypes.c_float, c_i32, c_vp]),
    "moe_permute_noalloc": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp]),
    "moe_quantize_mxfp8": (c_i32, [c_vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, c_vp, c_vp,
                                   ctypes.c_int64, c_vp]),
    "moe_permute_mxfp8": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                  c_vp, ctypes.c_size_t, c_vp]),
    "moe_grouped_ffn_mxfp8": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, c_vp, c_vp, c_vp, c_vp,
                                      ctypes.POINTER(MoeExpertWeightsMx), ctypes.POINTER(MoeFfnSaved), c_vp, c_vp,
                                      c_vp, ctypes.c_size_t, c_vp]),
    "moe_quantize_fp8_tile": (c_i32, [c_vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, c_vp, c_vp, c_vp]),
    "moe_grouped_ffn_fp8w": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, c_vp, c_vp, ctypes.POINTER(MoeExpertWeightsMx),
                                     ctypes.POINTER(MoeFfnSaved), c_vp, c_vp, c_vp, ctypes.c_size_t, c_vp]),
    "moe_backward_fp8w": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, ctypes.POINTER(MoeExpertWeightsMx),
                                  ctypes.POINTER(MoeFwdState), c_vp, ctypes.POINTER(MoeGrads), c_vp,
                                  ctypes.c_size_t, c_vp]),
    "moe_permute_capacity": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, c_vp, c_vp, ctypes.c_double, c_vp, c_vp, c_vp,
                                     c_vp, c_vp, c_vp, c_vp, c_vp, ctypes.c_size_t, c_vp]),
    "moe_aux_loss": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, c_vp, ctypes.c_float, c_vp, c_vp, c_vp,
                             ctypes.c_size_t, c_vp]),
    "moe_monitor_stats": (c_i32, [c_i32, c_vp, c_i32, c_vp, c_vp]),
    "moe_quantize_mxfp8_t": (c_i32, [c_vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, c_vp, c_vp,
                                     ctypes.c_int64, c_vp]),
    "moe_backward_mxfp8": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, ctypes.POINTER(MoeExpertWeightsMx),
                                   ctypes.POINTER(MoeFwdState), c_vp, ctypes.POINTER(MoeGrads), c_vp,
                                   ctypes.c_size_t, c_vp]),
    "moe_timing_enable": (c_i32, [c_i32]),
    "moe_timing_read": (c_i32, [c_i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64),
                                ctypes.POINTER(ctypes.c_int64)]),
    "moe_timing_disable": (c_i32, []),
    "moe_selftest_wait_timeout": (c_i32, [c_vp, ctypes.c_size_t, ctypes.c_uint64, c_i32, c_vp]),
    "moe_permute_maps": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, c_vp, c_vp, c_vp, c_vp, ctypes.c_size_t, c_vp]),
    "moe_grouped_ffn_gather": (c_i32, [ctypes.POINTER(MoeDesc), c_vp, c_vp, c_vp, ctypes.POINTER(MoeExpertWeights),
                                       ctypes.POINTER(MoeFfnSaved), c_vp, c_vp, c_vp, ctypes.c_size_t, c_vp]),
}

_LIB = None


def load(path: str | None = None):
    """Load libmoe.so (once) and attach the signatures."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or LIB
    if not os.path.exists(p):
        raise RuntimeError(f"libmoe.so is not built ({p}); run ragged_grouped_gemm_gb300.build.build()")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.moe_abi_version() != 1:
        raise RuntimeError("libmoe ABI version mismatch")
    if path is None:
        _LIB = lib
    return lib
