"""ctypes loader for libmxg.so: declares every C-ABI entry point of include/mxg.h.

Loading the library needs no GPU (the CUDA runtime is linked statically and
reaches the driver only on the first CUDA call).  A missing library raises;
there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmxg.so")

c_i32 = ctypes.c_int32
c_i64 = ctypes.c_int64
c_u64 = ctypes.c_uint64
c_size = ctypes.c_size_t
c_vp = ctypes.c_void_p


class MxOperandC(ctypes.Structure):
    """Mirror of ``mxg_mx_operand``."""
    _fields_ = [
        ("data", c_vp),
        ("scale", c_vp),
        ("rows", c_i64),
        ("cols", c_i64),
        ("ld", c_i64),
        ("scale_ld", c_i64),
        ("elem", c_i32),
        ("scale_layout", c_i32),
    ]


class BwOperandC(ctypes.Structure):
    """Mirror of ``mxg_bw_operand``."""
    _fields_ = [
        ("data", c_vp),
        ("scale", c_vp),
        ("rows", c_i64),
        ("cols", c_i64),
        ("ld", c_i64),
        ("scale_ld", c_i64),
        ("reserved0", c_i32),
        ("reserved1", c_i32),
    ]


# name -> (restype, argtypes); exactly the functions declared in include/mxg.h
SIGNATURES = {
    "mx_quantize_rowwise": (c_i32, [c_vp, c_i64, c_i64, c_i64, c_i32, c_vp, c_i64, c_vp, c_i64, c_vp]),
    "mx_quantize_colwise_segment_padded": (
        c_i32, [c_vp, c_i64, c_i64, c_i64, c_vp, c_i32, c_i32, c_i32, c_vp, c_i64, c_vp, c_i64,
                c_i64, c_vp, c_vp, c_vp]),
    "mx_quantize_dual_segment_padded": (
        c_i32, [c_vp, c_i64, c_i64, c_i64, c_vp, c_i32, c_i32, c_i32, c_vp, c_i64, c_vp, c_i64,
                c_vp, c_i64, c_vp, c_i64, c_i64, c_vp, c_vp, c_vp]),
    "mx_padded_rows_capacity": (c_i64, [c_i64, c_i32, c_i32]),
    "mx_packed_scale_bytes": (c_i64, [c_i64, c_i64, c_i32]),
    "mx_packed_colwise_scale_bytes": (c_i64, [c_i64, c_i64, c_i32]),
    "mx_quantize_colwise_segment_padded_packed": (
        c_i32, [c_vp, c_i64, c_i64, c_i64, c_vp, c_i32, c_i32, c_i32, c_vp, c_i64, c_vp, c_i64, c_i64, c_vp, c_vp,
                c_vp]),
    "mx_quantize_rowwise_packed": (c_i32, [c_vp, c_i64, c_i64, c_i64, c_i32, c_vp, c_i64, c_vp, c_i64, c_vp,
                                           c_i32, c_vp, c_vp]),
    "grouped_gemm_fwd": (
        c_i32, [ctypes.POINTER(MxOperandC), ctypes.POINTER(MxOperandC), c_vp, c_i32, c_i64, c_vp,
                c_i64, c_i32, c_vp, c_size, c_vp, c_vp]),
    "mx_gemm_dense": (
        c_i32, [ctypes.POINTER(MxOperandC), ctypes.POINTER(MxOperandC), c_vp, c_i64, c_i32, c_vp, c_size, c_vp,
                c_vp]),
    "grouped_gemm_dgrad": (
        c_i32, [ctypes.POINTER(MxOperandC), ctypes.POINTER(MxOperandC), c_vp, c_i32, c_vp, c_i64,
                c_i32, c_vp, c_size, c_vp, c_vp]),
    "grouped_gemm_wgrad": (
        c_i32, [ctypes.POINTER(MxOperandC), ctypes.POINTER(MxOperandC), c_vp, c_i32, c_i64, c_i32,
                c_vp, c_i32, c_i32, c_vp, c_size, c_vp, c_vp]),
    "grouped_gemm_fwd_noalloc": (
        c_i32, [ctypes.POINTER(MxOperandC), ctypes.POINTER(MxOperandC), c_vp, c_i32, c_i64, c_vp,
                c_i64, c_i32, c_vp, c_vp]),
    "mxg_gemm_workspace_size": (c_size, [c_i32, c_i32, c_i64, c_i64, c_i64, c_i32]),
    "bw_quantize_1x128": (c_i32, [c_vp, c_i64, c_i64, c_i64, c_vp, c_i64, c_vp, c_i64, c_vp]),
    "bw_quantize_128x128": (c_i32, [c_vp, c_i64, c_i64, c_i64, c_vp, c_i64, c_vp, c_vp, c_i64, c_vp,
                                    c_vp]),
    "bw_quantize_colwise_padded": (
        c_i32, [c_vp, c_i64, c_i64, c_i64, c_vp, c_i32, c_vp, c_i64, c_vp, c_i64, c_i64, c_vp, c_vp,
                c_vp]),
    "bw_quantize_1x128_pow2": (c_i32, [c_vp, c_i64, c_i64, c_i64, c_vp, c_i64, c_vp, c_i64, c_vp]),
    "bw_quantize_128x128_pow2": (c_i32, [c_vp, c_i64, c_i64, c_i64, c_vp, c_i64, c_vp, c_i64, c_vp,
                                         c_i64, c_vp, c_i64, c_vp]),
    "bw_quantize_colwise_padded_pow2": (
        c_i32, [c_vp, c_i64, c_i64, c_i64, c_vp, c_i32, c_vp, c_i64, c_vp, c_i64, c_i64, c_vp, c_vp,
                c_vp]),
    "bw_quantize_dual_padded": (
        c_i32, [c_vp, c_i64, c_i64, c_i64, c_vp, c_i32, c_vp, c_i64, c_vp, c_i64, c_vp, c_i64, c_vp, c_i64,
                c_i64, c_vp, c_vp, c_vp]),
    "bw_quantize_dual_padded_pow2": (
        c_i32, [c_vp, c_i64, c_i64, c_i64, c_vp, c_i32, c_vp, c_i64, c_vp, c_i64, c_vp, c_i64, c_vp, c_i64,
                c_i64, c_vp, c_vp, c_vp]),
    "bw_grouped_gemm_fwd": (
        c_i32, [ctypes.POINTER(BwOperandC), ctypes.POINTER(BwOperandC), c_vp, c_i32, c_i64, c_vp,
                c_i64, c_i32, c_vp, c_size, c_vp, c_vp]),
    "bw_grouped_gemm_dgrad": (
        c_i32, [ctypes.POINTER(BwOperandC), ctypes.POINTER(BwOperandC), c_vp, c_i32, c_vp, c_i64,
                c_i32, c_vp, c_size, c_vp, c_vp]),
    "bw_grouped_gemm_wgrad": (
        c_i32, [ctypes.POINTER(BwOperandC), ctypes.POINTER(BwOperandC), c_vp, c_i32, c_i64, c_vp,
                c_i32, c_i32, c_vp, c_size, c_vp, c_vp]),
    "bw_gemm_workspace_size": (c_size, [c_i32]),
    "mxg_check_status": (c_i32, [c_vp, c_vp]),
    "mxg_status_string": (ctypes.c_char_p, [c_i32]),
    "mxg_set_wait_timeout_ns": (None, [c_u64]),
    "mxg_get_wait_timeout_ns": (c_u64, []),
    "mxg_set_gemm_cta_group": (c_i32, [c_i32]),
    "mxg_get_gemm_cta_group": (c_i32, []),
    "mxg_diag_bounded_wait": (c_i32, [c_vp, c_u64, c_vp]),
    "mxg_version": (c_i32, []),
}

_lib = None


def load():
    """Load libmxg.so once and attach the signatures; raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
                "g.build()' or python fp8_bf16_mxfp4_gb300/build.py)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib
