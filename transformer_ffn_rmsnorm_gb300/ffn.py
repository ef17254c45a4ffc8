"""Python front end of the C ABI: argument marshalling only.

Each function takes torch tensors that already live on the GPU, passes their
device pointers and the current CUDA stream to the C entry point of the same
name, and raises ``FFNError`` on a non-OK status.  PyTorch supplies device
memory (outputs and workspace come from torch's allocator) and streams;
every step of the computation runs in the library's own kernels.
"""

from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _lib
from ._lib import (FFN_AUTO, FFN_BF16, FFN_F16, FFN_F32, FFN_GATEUP_FUSED,  # noqa: F401
                   FFN_GATEUP_UNFUSED, FFN_ACT_SINGLE, FFN_ACT_SPLIT, FFN_PATH_GEMM,
                   FFN_PATH_GEMV, FFN_PREPARED_WEIGHTS, FFN_RESIDUAL, FFN_DECODE_ONE_KERNEL,
                   Fp8Weight, Q4Weight, Q8Weight)

_DT = {torch.float32: FFN_F32, torch.float16: FFN_F16, torch.bfloat16: FFN_BF16}

_LIB = _lib.load()  # fail at import when the CUDA library is missing


class FFNError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = _lib.load()
        msg = lib.ffn_status_string(status).decode()
        super().__init__(f"{where}: {_lib.STATUS.get(status, status)} ({msg})")
        self.status = status


def _check(status: int, where: str):
    if status != 0:
        raise FFNError(status, where)


def _dtype(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def ffn_rmsnorm(x: torch.Tensor, g: torch.Tensor, eps: float, out: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    _need_cuda(x, g, out)
    d = x.shape[-1]
    rows = x.numel() // d if d else 0
    n = torch.empty_like(x) if out is None else out
    _check(_lib.load().ffn_rmsnorm(_ptr(x), _ptr(g), _ptr(n), rows, d, float(eps), _dtype(x),
                                   _stream(stream)), "ffn_rmsnorm")
    return n


def ffn_swiglu(gate: torch.Tensor, up: torch.Tensor, out: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    _need_cuda(gate, up, out)
    h = torch.empty_like(gate) if out is None else out
    _check(_lib.load().ffn_swiglu(_ptr(gate), _ptr(up), _ptr(h), gate.numel(), _dtype(gate),
                                  _stream(stream)), "ffn_swiglu")
    return h


def ffn_block_workspace_bytes(rows: int, d: int, ffn: int, dtype: torch.dtype, flags: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.load().ffn_block_workspace_bytes(rows, d, ffn, _DT[dtype], flags, ctypes.byref(out)),
           "ffn_block_workspace_bytes")
    return out.value


def workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def ffn_block_forward(x, g, w_gate, w_up, w_down, eps: float, flags: int = 0, out=None,
                      ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _need_cuda(x, g, w_gate, w_up, w_down, out, ws)
    d = x.shape[-1]
    rows = x.numel() // d
    ffn = w_gate.shape[0]
    y = torch.empty_like(x) if out is None else out
    if ws is None:   # (a passed workspace is checked against the need by the C side)
        ws = workspace(ffn_block_workspace_bytes(rows, d, ffn, x.dtype, flags), x.device)
    _check(_lib.load().ffn_block_forward(_ptr(x), _ptr(g), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                         _ptr(y), rows, d, ffn, float(eps), _dtype(x), flags,
                                         _ptr(ws), ws.numel(), _stream(stream)), "ffn_block_forward")
    return y


def ffn_block_forward_chained(x, g, w_gate, w_up, w_down, eps: float, flags: int = 0, x_sumsq=None,
                              y_sumsq: bool = True, out=None, ss_out=None, ws: torch.Tensor | None = None,
                              stream=None):
    """ffn_block_forward that takes each row's sum of squares of x (x_sumsq,
    fp32 [rows], or None) and returns (y, y_sumsq): the rows' sums of squares
    of the stored y (None unless y_sumsq)."""
    _need_cuda(x, g, w_gate, w_up, w_down, out, ws, x_sumsq, ss_out)
    d = x.shape[-1]
    rows = x.numel() // d
    ffn = w_gate.shape[0]
    y = torch.empty_like(x) if out is None else out
    ss = None
    if y_sumsq:
        ss = torch.empty(rows, dtype=torch.float32, device=x.device) if ss_out is None else ss_out
    if ws is None:
        ws = workspace(ffn_block_workspace_bytes(rows, d, ffn, x.dtype, flags), x.device)
    _check(_lib.load().ffn_block_forward_chained(_ptr(x), _ptr(x_sumsq), _ptr(g), _ptr(w_gate), _ptr(w_up),
                                                 _ptr(w_down), _ptr(y), _ptr(ss), rows, d, ffn, float(eps),
                                                 _dtype(x), flags, _ptr(ws), ws.numel(), _stream(stream)),
           "ffn_block_forward_chained")
    return y, ss


def ffn_block_host_workspace_bytes(rows: int, d: int, ffn: int, dtype, flags: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.load().ffn_block_host_workspace_bytes(rows, d, ffn, _DT[dtype], flags, ctypes.byref(out)),
           "ffn_block_host_workspace_bytes")
    return out.value


def ffn_block_forward_host(x_host, g, w_gate, w_up, w_down, eps: float, flags: int = 0, out=None,
                           ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The block with x and y in host memory (page-locked tensors overlap their
    copies with the compute); weights, g and the workspace on the device.
    Returns y on the host once `stream` (default: the current one) has passed
    the call; synchronise it before reading."""
    _need_cuda(g, w_gate, w_up, w_down, ws)
    if x_host.is_cuda or (out is not None and out.is_cuda):
        raise ValueError("x_host and out must be host tensors")
    if not x_host.is_contiguous() or (out is not None and not out.is_contiguous()):
        raise ValueError("x_host and out must be contiguous")
    d = x_host.shape[-1]
    rows = x_host.numel() // d
    ffn = w_gate.shape[0]
    y = torch.empty(x_host.shape, dtype=x_host.dtype, pin_memory=True) if out is None else out
    if ws is None:
        ws = workspace(ffn_block_host_workspace_bytes(rows, d, ffn, x_host.dtype, flags), g.device)
    _check(_lib.load().ffn_block_forward_host(_ptr(x_host), _ptr(g), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                              _ptr(y), rows, d, ffn, float(eps), _dtype(x_host), flags,
                                              _ptr(ws), ws.numel(), _stream(stream)), "ffn_block_forward_host")
    return y


def ffn_prepare_weights(w: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One-time re-encoding of a bf16/fp16 weight for FFN_PREPARED_WEIGHTS
    (fp16 values of w * 2^8)."""
    _need_cuda(w, out)
    dst = torch.empty(w.shape, dtype=torch.float16, device=w.device) if out is None else out
    _check(_lib.load().ffn_prepare_weights(_ptr(w), _ptr(dst), w.numel(), _dtype(w), _stream(stream)),
           "ffn_prepare_weights")
    return dst


def ffn_prepare_weights_fp8(w, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Prepared fp16 weights (values of e4m3 * row scale * 2^8) from a
    (codes [out, in], scales [out]) pair, for FFN_PREPARED_WEIGHTS."""
    codes, _ = w
    o, i = codes.shape
    dst = torch.empty((o, i), dtype=torch.float16, device=codes.device) if out is None else out
    _need_cuda(dst)
    _check(_lib.load().ffn_prepare_weights_fp8(_fp8(w), _ptr(dst), o, i, _stream(stream)), "ffn_prepare_weights_fp8")
    return dst


def ffn_prepare_weights_q4(w, inn: int, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Prepared fp16 weights (values of (u - 8) * s * 2^8) from a Q4 (qs,
    scales) pair in the device layout; `inn` is the input dimension."""
    qs, _ = w
    o = qs.shape[0]
    dst = torch.empty((o, inn), dtype=torch.float16, device=qs.device) if out is None else out
    _need_cuda(dst)
    _check(_lib.load().ffn_prepare_weights_q4(_q4(w), _ptr(dst), o, inn, _stream(stream)), "ffn_prepare_weights_q4")
    return dst


def ffn_block_q4_workspace_bytes(rows: int, d: int, ffn: int) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.load().ffn_block_q4_workspace_bytes(rows, d, ffn, ctypes.byref(out)),
           "ffn_block_q4_workspace_bytes")
    return out.value


def _q4(w):
    qs, sc = w
    _need_cuda(qs, sc)
    return Q4Weight(qs.data_ptr(), sc.data_ptr())


def ffn_block_forward_q4(x, g, w_gate, w_up, w_down, ffn: int, eps: float, flags: int = 0,
                         out=None, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """``w_*`` are (qs uint8, scales int16/uint16-bits) CUDA tensor pairs in the
    device layout of include/ffn.h."""
    _need_cuda(x, g, out, ws)
    d = x.shape[-1]
    rows = x.numel() // d
    y = torch.empty_like(x) if out is None else out
    if ws is None:
        ws = workspace(ffn_block_q4_workspace_bytes(rows, d, ffn), x.device)
    _check(_lib.load().ffn_block_forward_q4(_ptr(x), _ptr(g), _q4(w_gate), _q4(w_up), _q4(w_down),
                                            _ptr(y), rows, d, ffn, float(eps), flags, _ptr(ws),
                                            ws.numel(), _stream(stream)), "ffn_block_forward_q4")
    return y


def ffn_block_fp8_workspace_bytes(rows: int, d: int, ffn: int) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.load().ffn_block_fp8_workspace_bytes(rows, d, ffn, ctypes.byref(out)),
           "ffn_block_fp8_workspace_bytes")
    return out.value


def _fp8(w):
    codes, sc = w
    _need_cuda(codes, sc)
    if codes.element_size() != 1 or sc.dtype != torch.float32:
        raise TypeError("e4m3 weights are (1-byte codes, float32 row scales)")
    return Fp8Weight(codes.data_ptr(), sc.data_ptr())


def ffn_block_forward_fp8(x, g, w_gate, w_up, w_down, eps: float, flags: int = 0,
                          out=None, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """``w_*`` are (codes, scales) CUDA tensor pairs: e4m3 codes [out, in]
    (uint8 or torch.float8_e4m3fn) and float32 row scales [out]."""
    _need_cuda(x, g, out, ws)
    d = x.shape[-1]
    rows = x.numel() // d
    ffn = w_gate[0].shape[0]
    y = torch.empty_like(x) if out is None else out
    if ws is None:
        ws = workspace(ffn_block_fp8_workspace_bytes(rows, d, ffn), x.device)
    _check(_lib.load().ffn_block_forward_fp8(_ptr(x), _ptr(g), _fp8(w_gate), _fp8(w_up), _fp8(w_down),
                                             _ptr(y), rows, d, ffn, float(eps), flags, _ptr(ws),
                                             ws.numel(), _stream(stream)), "ffn_block_forward_fp8")
    return y


def ffn_block_q8_workspace_bytes(rows: int, d: int, ffn: int) -> int:
    out = ctypes.c_size_t(0)
    _check(_lib.load().ffn_block_q8_workspace_bytes(rows, d, ffn, ctypes.byref(out)),
           "ffn_block_q8_workspace_bytes")
    return out.value


def _q8(w):
    codes, sc = w
    _need_cuda(codes, sc)
    if codes.element_size() != 1 or sc.element_size() != 2:
        raise TypeError("Q8_0 weights are (1-byte codes, 2-byte fp16 scale bits)")
    return Q8Weight(codes.data_ptr(), sc.data_ptr())


def ffn_block_forward_q8(x, g, w_gate, w_up, w_down, eps: float, flags: int = 0,
                         out=None, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """``w_*`` are (codes int8 [out, in], scales [out, in/32] fp16 or their
    int16 bits) CUDA tensor pairs."""
    _need_cuda(x, g, out, ws)
    d = x.shape[-1]
    rows = x.numel() // d
    ffn = w_gate[0].shape[0]
    y = torch.empty_like(x) if out is None else out
    if ws is None:
        ws = workspace(ffn_block_q8_workspace_bytes(rows, d, ffn), x.device)
    _check(_lib.load().ffn_block_forward_q8(_ptr(x), _ptr(g), _q8(w_gate), _q8(w_up), _q8(w_down),
                                            _ptr(y), rows, d, ffn, float(eps), flags, _ptr(ws),
                                            ws.numel(), _stream(stream)), "ffn_block_forward_q8")
    return y


def ffn_prepare_weights_q8(w, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Prepared fp16 weights (values of q * s * 2^8) from a Q8_0 (codes,
    scales) pair, for FFN_PREPARED_WEIGHTS."""
    codes, _ = w
    o, i = codes.shape
    dst = torch.empty((o, i), dtype=torch.float16, device=codes.device) if out is None else out
    _need_cuda(dst)
    _check(_lib.load().ffn_prepare_weights_q8(_q8(w), _ptr(dst), o, i, _stream(stream)), "ffn_prepare_weights_q8")
    return dst


def ffn_q4_pack_host(q: np.ndarray, scales_bits: np.ndarray):
    """Host packer: int8 q [out, in] in [-8, 7] and fp16 scale bits [out, in/32]
    into the device layout (rows of ceil(in/128) 64-byte groups, 4 scales a
    group)."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    s = np.ascontiguousarray(scales_bits).view(np.uint16)
    out, inn = q.shape
    ngrp = -(-inn // 128)
    qs = np.empty((out, 64 * ngrp), dtype=np.uint8)
    so = np.empty((out, 4 * ngrp), dtype=np.uint16)
    _check(_lib.load().ffn_q4_pack_host(q.ctypes.data, s.ctypes.data, out, inn, qs.ctypes.data,
                                        so.ctypes.data), "ffn_q4_pack_host")
    return qs, so


def ffn_device_status():
    _check(_lib.load().ffn_device_status(), "ffn_device_status")


def ffn_selftest_bounded_wait(limit_ns: int = 2_000_000, stream=None):
    """Launch the bounded-wait self test: a wait that nothing completes gives
    up after limit_ns and the next ffn_device_status() raises FFN_ERR_TIMEOUT."""
    _check(_lib.load().ffn_selftest_bounded_wait(int(limit_ns), _stream(stream)), "ffn_selftest_bounded_wait")


def ffn_launch_count() -> int:
    return int(_lib.load().ffn_launch_count())


class KernelTimer:
    """Per-kernel device time from CUDA events recorded around each launch."""

    def __init__(self):
        self.lib = _lib.load()

    def __enter__(self):
        _check(self.lib.ffn_timing_reset(), "ffn_timing_reset")
        _check(self.lib.ffn_timing_enable(1), "ffn_timing_enable")
        return self

    def __exit__(self, *exc):
        self.lib.ffn_timing_enable(0)
        return False

    def read(self) -> dict:
        _check(self.lib.ffn_timing_collect(), "ffn_timing_collect")
        res = {}
        for k in range(self.lib.ffn_kernel_kinds()):
            n = ctypes.c_uint64(0)
            ms = ctypes.c_double(0.0)
            _check(self.lib.ffn_timing_read(k, ctypes.byref(n), ctypes.byref(ms)), "ffn_timing_read")
            if n.value:
                res[self.lib.ffn_kernel_name(k).decode()] = (int(n.value), float(ms.value))
        return res
