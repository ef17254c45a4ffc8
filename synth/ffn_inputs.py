"""Seeded synthetic inputs for the pre-norm SwiGLU FFN block.

Every tensor comes from its own numpy ``PCG64`` stream, keyed by
``SeedSequence([seed, tensor_id])``.  Values are drawn in float64 and then
rounded to their storage type:

* ``f32``  -- round to nearest even (numpy ``astype(float32)``);
* ``f16``  -- round to nearest even (numpy ``astype(float16)``);
* ``bf16`` -- round to float32, then to bfloat16 by round to nearest even.
  bfloat16 arrays are returned as ``uint16`` bit patterns.

The workloads below follow the five synthetic configurations the FFN
block is measured on (shapes, value distributions, eps).  ``N(0, v)``
is read as mean 0 and *variance* v, which gives unit-scale outputs.

The Q4 weight format is a data layout, so its packer lives here too; it
performs no arithmetic of the method.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np

__all__ = [
    "BlockConfig", "NormConfig", "SwigluConfig", "Q4Config",
    "C1_TINY_F32", "C2A_RMSNORM_F16", "C2B_SWIGLU_F16", "C3_DECODE_BF16",
    "C4_PREFILL_BF16", "C5_DECODE_Q4", "C8_BATCH_BF16", "CONFIGS",
    "stream", "normal", "round_to_storage", "make_block_inputs",
    "make_norm_inputs", "make_swiglu_inputs", "make_q4_inputs", "pack_q4",
    "q4_canonical_bytes", "TENSOR_IDS", "Fp8Config", "C6_DECODE_FP8", "make_fp8_inputs", "to_e4m3",
    "Q8Config", "C7_DECODE_Q8", "make_q8_inputs",
]

# Tensor ids inside one seed.  Each id owns an independent stream.
TENSOR_IDS = {
    "x": 0, "g": 1, "w_gate": 2, "w_up": 3, "w_down": 4,
    "q_gate": 5, "q_up": 6, "q_down": 7,
    "s_gate": 8, "s_up": 9, "s_down": 10,
    "gate": 11, "up": 12,
    "f8_gate": 13, "f8_up": 14, "f8_down": 15, "f8s_gate": 16, "f8s_up": 17, "f8s_down": 18,
    "q8_gate": 19, "q8_up": 20, "q8_down": 21, "q8s_gate": 22, "q8s_up": 23, "q8s_down": 24,
}

_CHUNK = 1 << 22


def stream(seed: int, tensor: str | int) -> np.random.Generator:
    tid = TENSOR_IDS[tensor] if isinstance(tensor, str) else int(tensor)
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), tid])))


def _f32_to_bf16_bits(a32: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest even); return uint16 bits."""
    b = np.ascontiguousarray(a32, dtype=np.float32).view(np.uint32)
    nan = (b & 0x7F800000) == 0x7F800000
    nan &= (b & 0x007FFFFF) != 0
    lsb = (b >> 16) & 1
    r = ((b.astype(np.uint64) + 0x7FFF + lsb) >> 16).astype(np.uint16)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def round_to_storage(a64: np.ndarray, dtype: str) -> np.ndarray:
    """Round a float64 array to its storage type (see module docstring)."""
    if dtype == "f32":
        return a64.astype(np.float32)
    if dtype == "f16":
        return a64.astype(np.float16)
    if dtype == "bf16":
        return _f32_to_bf16_bits(a64.astype(np.float32))
    raise ValueError(f"unknown storage dtype {dtype!r}")


def _storage_empty(shape, dtype: str) -> np.ndarray:
    npdt = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[dtype]
    return np.empty(shape, dtype=npdt)


def normal(shape, mean: float, std: float, seed: int, tensor, dtype: str) -> np.ndarray:
    """mean + std * N(0,1) drawn in float64, rounded once to ``dtype``."""
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    out = _storage_empty((n,), dtype)
    rng = stream(seed, tensor)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        v = rng.standard_normal(hi - lo)
        if std != 1.0:
            v *= std
        if mean != 0.0:
            v += mean
        out[lo:hi] = round_to_storage(v, dtype)
    return out.reshape(shape)


# --------------------------------------------------------------------------
# Workload descriptions
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class BlockConfig:
    name: str
    rows: int
    d: int
    ffn: int
    eps: float
    dtype: str          # storage type of x, g, weights, y


@dataclass(frozen=True)
class NormConfig:
    name: str
    rows: int
    d: int
    eps: float
    dtype: str


@dataclass(frozen=True)
class SwigluConfig:
    name: str
    rows: int
    cols: int
    dtype: str
    std: float


@dataclass(frozen=True)
class Q4Config:
    name: str
    rows: int
    d: int
    ffn: int
    eps: float


C1_TINY_F32 = BlockConfig("tiny_f32_64x256x704", 64, 256, 704, 1e-6, "f32")
C2A_RMSNORM_F16 = NormConfig("rmsnorm_f16_16384x4096", 16384, 4096, 1e-5, "f16")
C2B_SWIGLU_F16 = SwigluConfig("swiglu_f16_16384x11008", 16384, 11008, "f16", math.sqrt(2.0))
C3_DECODE_BF16 = BlockConfig("decode_bf16_8x4096x14336", 8, 4096, 14336, 1e-5, "bf16")
C4_PREFILL_BF16 = BlockConfig("prefill_bf16_4096x4096x11008", 4096, 4096, 11008, 1e-6, "bf16")
# a batch of 128 decode tokens through the decode layer shape (one row block)
C8_BATCH_BF16 = BlockConfig("batch_bf16_128x4096x14336", 128, 4096, 14336, 1e-5, "bf16")
C5_DECODE_Q4 = Q4Config("decode_q4_8x5120x17408", 8, 5120, 17408, 1e-6)


@dataclass(frozen=True)
class Fp8Config:
    name: str
    rows: int
    d: int
    ffn: int
    eps: float


# the bf16 decode shape with e4m3 weights (per-row float scales)
C6_DECODE_FP8 = Fp8Config("decode_fp8_8x4096x14336", 8, 4096, 14336, 1e-5)

CONFIGS = {
    "c1": C1_TINY_F32, "c2a": C2A_RMSNORM_F16, "c2b": C2B_SWIGLU_F16,
    "c3": C3_DECODE_BF16, "c4": C4_PREFILL_BF16, "c5": C5_DECODE_Q4, "c6": C6_DECODE_FP8,
    "c8": C8_BATCH_BF16,
}


def make_block_inputs(cfg: BlockConfig, seed: int = 0, rows: int | None = None,
                      d: int | None = None, ffn: int | None = None) -> dict:
    """x~N(0,1), g=1+0.1*N(0,1), W_gate/W_up [ffn x d] and W_down [d x ffn]
    ~N(0, 1/fan_in); all rounded to ``cfg.dtype``.  Overrides allow smaller
    instances with the same recipe."""
    cfg = replace(cfg, rows=rows if rows is not None else cfg.rows,
                  d=d if d is not None else cfg.d,
                  ffn=ffn if ffn is not None else cfg.ffn)
    M, D, F, dt = cfg.rows, cfg.d, cfg.ffn, cfg.dtype
    return {
        "cfg": cfg,
        "x": normal((M, D), 0.0, 1.0, seed, "x", dt),
        "g": normal((D,), 1.0, 0.1, seed, "g", dt),
        "w_gate": normal((F, D), 0.0, 1.0 / math.sqrt(D), seed, "w_gate", dt),
        "w_up": normal((F, D), 0.0, 1.0 / math.sqrt(D), seed, "w_up", dt),
        "w_down": normal((D, F), 0.0, 1.0 / math.sqrt(F), seed, "w_down", dt),
    }


def make_norm_inputs(cfg: NormConfig, seed: int = 0, rows: int | None = None,
                     d: int | None = None) -> dict:
    cfg = replace(cfg, rows=rows if rows is not None else cfg.rows,
                  d=d if d is not None else cfg.d)
    return {
        "cfg": cfg,
        "x": normal((cfg.rows, cfg.d), 0.0, 1.0, seed, "x", cfg.dtype),
        "g": normal((cfg.d,), 1.0, 0.1, seed, "g", cfg.dtype),
    }


def make_swiglu_inputs(cfg: SwigluConfig, seed: int = 0, rows: int | None = None,
                       cols: int | None = None) -> dict:
    cfg = replace(cfg, rows=rows if rows is not None else cfg.rows,
                  cols=cols if cols is not None else cfg.cols)
    shape = (cfg.rows, cfg.cols)
    return {
        "cfg": cfg,
        "gate": normal(shape, 0.0, cfg.std, seed, "gate", cfg.dtype),
        "up": normal(shape, 0.0, cfg.std, seed, "up", cfg.dtype),
    }


# --------------------------------------------------------------------------
# Q4 weights
# --------------------------------------------------------------------------

def q4_canonical_bytes(q: np.ndarray) -> np.ndarray:
    """Canonical 16 nibble bytes per 32-weight block.

    ``q`` is int8 [out, in] with values in [-8, 7].  Each weight is stored
    offset-binary, u = q + 8.  Byte i (0..15) of a block holds u[i] in its
    low nibble and u[i + 16] in its high nibble.  Returns uint8
    [out, in/32, 16]."""
    out, inn = q.shape
    if inn % 32:
        raise ValueError("Q4 rows must hold whole 32-weight blocks")
    if q.min(initial=0) < -8 or q.max(initial=0) > 7:
        raise ValueError("Q4 values must lie in [-8, 7]")
    u = (q.astype(np.int16) + 8).astype(np.uint8).reshape(out, inn // 32, 32)
    return (u[:, :, :16] | (u[:, :, 16:] << 4)).astype(np.uint8)


def pack_q4(q: np.ndarray, scales_f16: np.ndarray):
    """Pack int8 Q4 values and fp16 block scales into the device layout.

    Device layout of ``qs`` (uint8): blocks are grouped four at a time along
    the input dimension; inside a group of 64 bytes, offset 16*t + 4*b + e
    holds canonical byte 4*t + e of block b of the group (t, b, e in 0..3).
    A row holds ceil(in/128) groups (in/2 bytes when in % 128 == 0); the
    blocks of a last, partial group past in/32 are zero bytes.  ``scales``:
    [out, 4*ceil(in/128)] fp16 bits, zero past in/32.  Requires
    ``in % 32 == 0``."""
    out, inn = q.shape
    if inn % 32:
        raise ValueError("the Q4 device layout needs in % 32 == 0")
    nb, ngrp = inn // 32, -(-inn // 128)
    cb = np.zeros((out, 4 * ngrp, 16), dtype=np.uint8)
    cb[:, :nb] = q4_canonical_bytes(q)                    # [out, 4G, 16]
    g = cb.reshape(out, ngrp, 4, 4, 4)                    # [o, G, b, t, e]
    qs = np.ascontiguousarray(g.transpose(0, 1, 3, 2, 4)).reshape(out, 64 * ngrp)
    sc16 = np.ascontiguousarray(np.asarray(scales_f16, dtype=np.float16)).view(np.uint16)
    if sc16.shape != (out, nb):
        raise ValueError("scales must be [out, in/32]")
    sc = np.zeros((out, 4 * ngrp), dtype=np.uint16)
    sc[:, :nb] = sc16
    return qs, sc


def make_q4_inputs(cfg: Q4Config, seed: int = 0, rows: int | None = None,
                   d: int | None = None, ffn: int | None = None) -> dict:
    """x~N(0,1) bf16, g=1+0.1*N(0,1) bf16, Q4 weights with q~U{-8..7} and
    fp16 scales |N(0,1)| / (8*sqrt(fan_in))."""
    cfg = replace(cfg, rows=rows if rows is not None else cfg.rows,
                  d=d if d is not None else cfg.d,
                  ffn=ffn if ffn is not None else cfg.ffn)
    M, D, F = cfg.rows, cfg.d, cfg.ffn
    res = {"cfg": cfg,
           "x": normal((M, D), 0.0, 1.0, seed, "x", "bf16"),
           "g": normal((D,), 1.0, 0.1, seed, "g", "bf16")}
    for name, (o, i) in (("gate", (F, D)), ("up", (F, D)), ("down", (D, F))):
        q = stream(seed, "q_" + name).integers(-8, 8, size=(o, i), dtype=np.int8)
        s64 = np.abs(stream(seed, "s_" + name).standard_normal((o, i // 32))) / (8.0 * math.sqrt(i))
        s16 = s64.astype(np.float16)
        qs, sc = pack_q4(q, s16)
        res["q_" + name] = q
        res["s_" + name] = s16
        res["qs_" + name] = qs
        res["sc_" + name] = sc
    return res


def to_e4m3(v: np.ndarray) -> np.ndarray:
    """e4m3 ("fn") codes of float values, round to nearest even (a library
    conversion; values must lie within +-448)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def make_fp8_inputs(cfg: Fp8Config, seed: int = 0, rows: int | None = None,
                    d: int | None = None, ffn: int | None = None) -> dict:
    """x~N(0,1) bf16, g=1+0.1*N(0,1) bf16, weights as e4m3 codes of
    16*N(0,1) with float32 row scales (1 + 0.1*N(0,1)) / (16*sqrt(fan_in)),
    i.e. weights ~N(0, 1/fan_in) as in the other block workloads."""
    cfg = replace(cfg, rows=rows if rows is not None else cfg.rows,
                  d=d if d is not None else cfg.d,
                  ffn=ffn if ffn is not None else cfg.ffn)
    M, D, F = cfg.rows, cfg.d, cfg.ffn
    res = {"cfg": cfg,
           "x": normal((M, D), 0.0, 1.0, seed, "x", "bf16"),
           "g": normal((D,), 1.0, 0.1, seed, "g", "bf16")}
    for name, (o, i) in (("gate", (F, D)), ("up", (F, D)), ("down", (D, F))):
        v = np.clip(16.0 * stream(seed, "f8_" + name).standard_normal((o, i)), -448.0, 448.0)
        res["c_" + name] = to_e4m3(v)
        sc = (1.0 + 0.1 * stream(seed, "f8s_" + name).standard_normal(o)) / (16.0 * math.sqrt(i))
        res["s_" + name] = sc.astype(np.float32)
    return res


# ------------------------------------------------------------------ Q8_0
@dataclass(frozen=True)
class Q8Config:
    name: str
    rows: int
    d: int
    ffn: int
    eps: float


# the bf16 decode shape with Q8_0 weights (int8 codes, an fp16 scale per 32)
C7_DECODE_Q8 = Q8Config("decode_q8_8x4096x14336", 8, 4096, 14336, 1e-5)


def make_q8_inputs(cfg: Q8Config, seed: int = 0, rows: int | None = None,
                   d: int | None = None, ffn: int | None = None) -> dict:
    """x~N(0,1) bf16, g=1+0.1*N(0,1) bf16, weights as int8 codes
    clip(round(32*N(0,1)), -128, 127) with fp16 block scales
    (1 + 0.1*N(0,1)) / (32*sqrt(fan_in)), i.e. weights ~N(0, 1/fan_in) as in
    the other block workloads.  Scales are returned as uint16 bit patterns."""
    cfg = replace(cfg, rows=rows if rows is not None else cfg.rows,
                  d=d if d is not None else cfg.d,
                  ffn=ffn if ffn is not None else cfg.ffn)
    M, D, F = cfg.rows, cfg.d, cfg.ffn
    res = {"cfg": cfg,
           "x": normal((M, D), 0.0, 1.0, seed, "x", "bf16"),
           "g": normal((D,), 1.0, 0.1, seed, "g", "bf16")}
    for name, (o, i) in (("gate", (F, D)), ("up", (F, D)), ("down", (D, F))):
        q = np.clip(np.rint(32.0 * stream(seed, "q8_" + name).standard_normal((o, i))), -128, 127)
        res["q8_" + name] = q.astype(np.int8)
        sc = (1.0 + 0.1 * stream(seed, "q8s_" + name).standard_normal((o, i // 32))) / (32.0 * math.sqrt(i))
        res["q8s_" + name] = sc.astype(np.float16).view(np.uint16)
    return res
