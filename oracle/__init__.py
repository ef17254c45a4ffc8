"""TEST INFRASTRUCTURE -- the float64 CPU oracle for the pre-norm SwiGLU FFN block.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package never imports the CUDA library: the two share no code.  Inputs come
from the seeded generators in ``synth``; this wrapper only widens stored
values to float64 (exactly) and hands them to the C routines in
``ffn_oracle.c``, which carry the arithmetic and its citations.

Parity pins: every routine here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, brute force on tiny inputs, the Q4 layout against
the generator's integers); see also ``tests/test_oracle_mutants.py``, which
plants plausible mistakes into a copy of the C source and checks that a pin
catches each one.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "ffn_oracle.c")
LIBPATH = os.path.join(HERE, "liboracle_ffn.so")

_D = ctypes.POINTER(ctypes.c_double)


def build(source: str = SOURCE, out: str = LIBPATH, cc: str = "cc") -> str:
    """Compile the oracle with plain IEEE double semantics."""
    cmd = [cc, "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-o", out, source, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    return out


def _stale(lib: str, src: str) -> bool:
    return (not os.path.exists(lib)) or os.path.getmtime(lib) < os.path.getmtime(src)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Stored values -> float64, exactly.  bf16 arrive as uint16 bit patterns."""
    if dtype == "bf16":
        u = np.ascontiguousarray(a, dtype=np.uint16).astype(np.uint32) << 16
        return u.view(np.float32).astype(np.float64)
    if dtype in ("f16", "f32"):
        return np.asarray(a).astype(np.float64)
    raise ValueError(dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_D)


class Oracle:
    """ctypes front end of one compiled copy of the oracle."""

    def __init__(self, libpath: str | None = None, source: str = SOURCE):
        if libpath is None:
            libpath = LIBPATH
            if _stale(libpath, source):
                build(source, libpath)
        self.libpath = libpath
        L = ctypes.CDLL(libpath)
        L.oracle_silu.restype = ctypes.c_double
        L.oracle_silu.argtypes = [ctypes.c_double]
        L.oracle_half_to_double.restype = ctypes.c_double
        L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_rmsnorm.restype = None
        L.oracle_rmsnorm.argtypes = [_D, _D, _D, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_double, ctypes.c_int]
        L.oracle_row_sumsq.restype = None
        L.oracle_row_sumsq.argtypes = [_D, _D, ctypes.c_int64, ctypes.c_int64]
        L.oracle_swiglu.restype = None
        L.oracle_swiglu.argtypes = [_D, _D, _D, ctypes.c_int64, ctypes.c_int]
        L.oracle_ffn_block.restype = ctypes.c_int
        L.oracle_ffn_block.argtypes = [_D, _D, _D, _D, _D, _D, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
                                       ctypes.c_int]
        L.oracle_q4_dequant.restype = None
        L.oracle_q4_dequant.argtypes = [ctypes.POINTER(ctypes.c_uint8),
                                        ctypes.POINTER(ctypes.c_uint16), _D,
                                        ctypes.c_int64, ctypes.c_int64]
        L.oracle_e4m3_to_double.restype = ctypes.c_double
        L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_q8_dequant.restype = None
        L.oracle_q8_dequant.argtypes = [ctypes.POINTER(ctypes.c_int8), ctypes.POINTER(ctypes.c_uint16), _D,
                                        ctypes.c_int64, ctypes.c_int64]
        L.oracle_fp8_dequant.restype = None
        L.oracle_fp8_dequant.argtypes = [ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(ctypes.c_float), _D,
                                         ctypes.c_int64, ctypes.c_int64]
        self.L = L

    # -- scalars ---------------------------------------------------------
    def silu(self, z: float) -> float:
        return self.L.oracle_silu(float(z))

    def half_to_double(self, bits: int) -> float:
        return self.L.oracle_half_to_double(int(bits) & 0xFFFF)

    def e4m3_to_double(self, code: int) -> float:
        return self.L.oracle_e4m3_to_double(int(code) & 0xFF)

    # -- arrays (float64 in, float64 out) --------------------------------
    def rmsnorm(self, x, g, eps: float, nthreads: int | None = None) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float64)
        g = np.ascontiguousarray(g, dtype=np.float64)
        rows, d = x.shape
        assert g.shape == (d,)
        n = np.empty_like(x)
        self.L.oracle_rmsnorm(_ptr(x), _ptr(g), _ptr(n), rows, d, float(eps),
                              nthreads or default_threads())
        return n

    def row_sumsq(self, y) -> np.ndarray:
        """Sum of squares of every row of y (the next RMSNorm's reduction)."""
        y = np.ascontiguousarray(y, dtype=np.float64)
        rows, d = y.shape
        ss = np.empty(rows, dtype=np.float64)
        self.L.oracle_row_sumsq(_ptr(y), _ptr(ss), rows, d)
        return ss

    def swiglu(self, gate, up, nthreads: int | None = None) -> np.ndarray:
        gate = np.ascontiguousarray(gate, dtype=np.float64)
        up = np.ascontiguousarray(up, dtype=np.float64)
        assert gate.shape == up.shape
        h = np.empty_like(gate)
        self.L.oracle_swiglu(_ptr(gate), _ptr(up), _ptr(h), gate.size,
                             nthreads or default_threads())
        return h

    def ffn_block(self, x, g, w_gate, w_up, w_down, eps: float,
                  nthreads: int | None = None, residual: bool = False) -> np.ndarray:
        """y = W_down (silu(W_gate n) * (W_up n)), n = RMSNorm(x); with
        ``residual``, y = x + that (the block's skip connection, added in
        float64)."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        g = np.ascontiguousarray(g, dtype=np.float64)
        w_gate = np.ascontiguousarray(w_gate, dtype=np.float64)
        w_up = np.ascontiguousarray(w_up, dtype=np.float64)
        w_down = np.ascontiguousarray(w_down, dtype=np.float64)
        rows, d = x.shape
        ffn = w_gate.shape[0]
        assert g.shape == (d,) and w_gate.shape == (ffn, d) and w_up.shape == (ffn, d)
        assert w_down.shape == (d, ffn)
        y = np.empty((rows, d), dtype=np.float64)
        rc = self.L.oracle_ffn_block(_ptr(x), _ptr(g), _ptr(w_gate), _ptr(w_up), _ptr(w_down),
                                     _ptr(y), rows, d, ffn, float(eps),
                                     nthreads or default_threads())
        if rc != 0:
            raise MemoryError("oracle scratch allocation failed")
        return x + y if residual else y

    def fp8_dequant(self, codes, scales, out: int, inn: int) -> np.ndarray:
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.float32)
        assert codes.size == out * inn and scales.size == out
        w = np.empty((out, inn), dtype=np.float64)
        self.L.oracle_fp8_dequant(codes.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
                                  scales.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), _ptr(w), out, inn)
        return w

    def fp8_block_from_inputs(self, inp: dict, rows=None, nthreads=None, residual=False) -> np.ndarray:
        """Oracle y for a ``synth.make_fp8_inputs`` dict, on weights the oracle
        dequantises itself from the e4m3 codes and row scales."""
        cfg = inp["cfg"]
        D, F = cfg.d, cfg.ffn
        wg = self.fp8_dequant(inp["c_gate"], inp["s_gate"], F, D)
        wu = self.fp8_dequant(inp["c_up"], inp["s_up"], F, D)
        wd = self.fp8_dequant(inp["c_down"], inp["s_down"], D, F)
        x = inp["x"] if rows is None else inp["x"][np.asarray(rows)]
        return self.ffn_block(widen(x, "bf16"), widen(inp["g"], "bf16"), wg, wu, wd, cfg.eps, nthreads, residual)

    def q4_dequant(self, qs, scales, out: int, inn: int) -> np.ndarray:
        qs = np.ascontiguousarray(qs, dtype=np.uint8)
        scales = np.ascontiguousarray(scales, dtype=np.uint16)
        ngrp = -(-inn // 128)   # groups of four blocks a row, the last one padded
        assert qs.size == out * ngrp * 64 and scales.size == out * ngrp * 4
        w = np.empty((out, inn), dtype=np.float64)
        self.L.oracle_q4_dequant(qs.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
                                 scales.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
                                 _ptr(w), out, inn)
        return w

    def q8_dequant(self, q, scales, out: int, inn: int) -> np.ndarray:
        q = np.ascontiguousarray(q, dtype=np.int8)
        scales = np.ascontiguousarray(scales).view(np.uint16)
        assert q.size == out * inn and scales.size == out * (inn // 32)
        w = np.empty((out, inn), dtype=np.float64)
        self.L.oracle_q8_dequant(q.ctypes.data_as(ctypes.POINTER(ctypes.c_int8)),
                                 scales.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), _ptr(w), out, inn)
        return w

    def q8_block_from_inputs(self, inp: dict, rows=None, nthreads=None, residual=False) -> np.ndarray:
        """Oracle y for a ``synth.make_q8_inputs`` dict, on weights the oracle
        dequantises itself from the codes and scale bits."""
        cfg = inp["cfg"]
        D, F = cfg.d, cfg.ffn
        wg = self.q8_dequant(inp["q8_gate"], inp["q8s_gate"], F, D)
        wu = self.q8_dequant(inp["q8_up"], inp["q8s_up"], F, D)
        wd = self.q8_dequant(inp["q8_down"], inp["q8s_down"], D, F)
        x = inp["x"] if rows is None else inp["x"][np.asarray(rows)]
        return self.ffn_block(widen(x, "bf16"), widen(inp["g"], "bf16"), wg, wu, wd, cfg.eps, nthreads, residual)

    # -- convenience: stored inputs -> float64 result --------------------
    def block_from_inputs(self, inp: dict, rows=None, nthreads=None, residual=False) -> np.ndarray:
        """Oracle y for a ``synth.make_block_inputs`` dict; ``rows`` selects a
        subset of token rows (rows are independent)."""
        dt = inp["cfg"].dtype
        x = inp["x"] if rows is None else inp["x"][np.asarray(rows)]
        return self.ffn_block(widen(x, dt), widen(inp["g"], dt), widen(inp["w_gate"], dt),
                              widen(inp["w_up"], dt), widen(inp["w_down"], dt),
                              inp["cfg"].eps, nthreads, residual)

    def q4_block_from_inputs(self, inp: dict, rows=None, nthreads=None, residual=False) -> np.ndarray:
        """Oracle y for a ``synth.make_q4_inputs`` dict, on weights the oracle
        dequantises itself from the packed bytes."""
        cfg = inp["cfg"]
        D, F = cfg.d, cfg.ffn
        wg = self.q4_dequant(inp["qs_gate"], inp["sc_gate"], F, D)
        wu = self.q4_dequant(inp["qs_up"], inp["sc_up"], F, D)
        wd = self.q4_dequant(inp["qs_down"], inp["sc_down"], D, F)
        x = inp["x"] if rows is None else inp["x"][np.asarray(rows)]
        return self.ffn_block(widen(x, "bf16"), widen(inp["g"], "bf16"), wg, wu, wd,
                              cfg.eps, nthreads, residual)


_default = None


def get() -> Oracle:
    """The oracle compiled from ``ffn_oracle.c`` (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
