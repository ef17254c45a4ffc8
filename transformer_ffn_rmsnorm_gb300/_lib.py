"""ctypes declarations of the C ABI in include/ffn.h (libffn_gb300.so).

Loading fails loudly when the library has not been built: there is no
fallback implementation behind these names.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIBPATH = os.path.join(HERE, "libffn_gb300.so")

c_void_p, c_int64, c_float, c_int, c_uint32, c_size_t = (
    ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_uint32, ctypes.c_size_t)

STATUS = {
    0: "FFN_OK", 1: "FFN_ERR_NULL", 2: "FFN_ERR_SHAPE", 3: "FFN_ERR_DTYPE", 4: "FFN_ERR_ALIGN",
    5: "FFN_ERR_WORKSPACE", 6: "FFN_ERR_ALIAS", 7: "FFN_ERR_CUDA", 8: "FFN_ERR_TIMEOUT",
    9: "FFN_ERR_FLAGS", 10: "FFN_ERR_RANGE",
}
FFN_OK, FFN_ERR_NULL, FFN_ERR_SHAPE, FFN_ERR_DTYPE, FFN_ERR_ALIGN = 0, 1, 2, 3, 4
FFN_ERR_WORKSPACE, FFN_ERR_ALIAS, FFN_ERR_CUDA, FFN_ERR_TIMEOUT, FFN_ERR_FLAGS = 5, 6, 7, 8, 9
FFN_ERR_RANGE = 10
FFN_F32, FFN_F16, FFN_BF16 = 0, 1, 2
FFN_AUTO, FFN_GATEUP_FUSED, FFN_GATEUP_UNFUSED, FFN_PATH_GEMM, FFN_PATH_GEMV = 0, 1, 2, 4, 8
FFN_ACT_SINGLE, FFN_ACT_SPLIT, FFN_PREPARED_WEIGHTS = 16, 32, 64
FFN_RESIDUAL, FFN_DECODE_ONE_KERNEL = 128, 256


class Q4Weight(ctypes.Structure):
    _fields_ = [("qs", c_void_p), ("scales", c_void_p)]


class Fp8Weight(ctypes.Structure):
    _fields_ = [("codes", c_void_p), ("scales", c_void_p)]


class Q8Weight(ctypes.Structure):
    _fields_ = [("codes", c_void_p), ("scales", c_void_p)]


# name -> (restype, argtypes), in the order of include/ffn.h
SIGNATURES = {
    "ffn_rmsnorm": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_float, c_int, c_void_p]),
    "ffn_swiglu": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int, c_void_p]),
    "ffn_block_workspace_bytes": (c_int, [c_int64, c_int64, c_int64, c_int, c_uint32,
                                          ctypes.POINTER(c_size_t)]),
    "ffn_block_forward": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                  c_int64, c_int64, c_int64, c_float, c_int, c_uint32, c_void_p,
                                  c_size_t, c_void_p]),
    "ffn_block_forward_chained": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                          c_void_p, c_int64, c_int64, c_int64, c_float, c_int, c_uint32,
                                          c_void_p, c_size_t, c_void_p]),
    "ffn_block_host_workspace_bytes": (c_int, [c_int64, c_int64, c_int64, c_int, c_uint32,
                                               ctypes.POINTER(c_size_t)]),
    "ffn_block_forward_host": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                       c_int64, c_int64, c_int64, c_float, c_int, c_uint32, c_void_p,
                                       c_size_t, c_void_p]),
    "ffn_block_q4_workspace_bytes": (c_int, [c_int64, c_int64, c_int64, ctypes.POINTER(c_size_t)]),
    "ffn_block_forward_q4": (c_int, [c_void_p, c_void_p, Q4Weight, Q4Weight, Q4Weight, c_void_p,
                                     c_int64, c_int64, c_int64, c_float, c_uint32, c_void_p,
                                     c_size_t, c_void_p]),
    "ffn_block_fp8_workspace_bytes": (c_int, [c_int64, c_int64, c_int64, ctypes.POINTER(c_size_t)]),
    "ffn_block_forward_fp8": (c_int, [c_void_p, c_void_p, Fp8Weight, Fp8Weight, Fp8Weight, c_void_p,
                                      c_int64, c_int64, c_int64, c_float, c_uint32, c_void_p,
                                      c_size_t, c_void_p]),
    "ffn_block_q8_workspace_bytes": (c_int, [c_int64, c_int64, c_int64, ctypes.POINTER(c_size_t)]),
    "ffn_block_forward_q8": (c_int, [c_void_p, c_void_p, Q8Weight, Q8Weight, Q8Weight, c_void_p,
                                     c_int64, c_int64, c_int64, c_float, c_uint32, c_void_p,
                                     c_size_t, c_void_p]),
    "ffn_block_forward_decode_static": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                                c_void_p, c_int64, c_int64, c_int64, c_float, c_int,
                                                c_void_p]),
    "ffn_prepare_weights": (c_int, [c_void_p, c_void_p, c_int64, c_int, c_void_p]),
    "ffn_prepare_weights_fp8": (c_int, [Fp8Weight, c_void_p, c_int64, c_int64, c_void_p]),
    "ffn_prepare_weights_q4": (c_int, [Q4Weight, c_void_p, c_int64, c_int64, c_void_p]),
    "ffn_prepare_weights_q8": (c_int, [Q8Weight, c_void_p, c_int64, c_int64, c_void_p]),
    "ffn_q4_pack_host": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_void_p, c_void_p]),
    "ffn_status_string": (ctypes.c_char_p, [c_int]),
    "ffn_device_status": (c_int, []),
    "ffn_selftest_bounded_wait": (c_int, [ctypes.c_uint64, c_void_p]),
    "ffn_launch_count": (ctypes.c_uint64, []),
    "ffn_timing_enable": (c_int, [c_int]),
    "ffn_timing_collect": (c_int, []),
    "ffn_timing_reset": (c_int, []),
    "ffn_kernel_kinds": (c_int, []),
    "ffn_kernel_name": (ctypes.c_char_p, [c_int]),
    "ffn_timing_read": (c_int, [c_int, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_double)]),
}

_lib = None


def load(path: str = LIBPATH) -> ctypes.CDLL:
    """The C library, with argument and result types declared."""
    global _lib
    if _lib is not None and path == LIBPATH:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(no fallback implementation exists)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == LIBPATH:
        _lib = lib
    return lib
