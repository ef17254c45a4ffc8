"""ffn_block_forward_fp8 on the GPU against the oracle, which decodes the e4m3
codes and applies the row scales itself (float64)."""

import numpy as np
import pytest

import synth
from gpu_util import assert_lowp, fp8_dev, to_dev, to_host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ffn():
    from transformer_ffn_rmsnorm_gb300 import ffn as m
    return m


def run_fp8(ffn, inp, flags=0):
    cfg = inp["cfg"]
    return ffn.ffn_block_forward_fp8(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"),
                                     fp8_dev(inp, "gate"), fp8_dev(inp, "up"), fp8_dev(inp, "down"),
                                     eps=cfg.eps, flags=flags)


def test_fp8_full_size(ffn, oracle_lib):
    """8 rows, d=4096, ffn=14336, e4m3 weights with row scales."""
    inp = synth.make_fp8_inputs(synth.C6_DECODE_FP8, seed=0)
    assert_lowp(to_host64(run_fp8(ffn, inp)), oracle_lib.fp8_block_from_inputs(inp))


@pytest.mark.parametrize("rows", [1, 3, 8, 9, 16, 20, 33])
def test_fp8_rows(ffn, oracle_lib, rows):
    """One and two token tiles, ragged tiles, and more than 16 rows (groups)."""
    inp = synth.make_fp8_inputs(synth.C6_DECODE_FP8, seed=rows, rows=rows, d=1024, ffn=2816)
    assert_lowp(to_host64(run_fp8(ffn, inp)), oracle_lib.fp8_block_from_inputs(inp))


@pytest.mark.parametrize("d,ffn_", [(256, 256), (768, 1280), (4096, 2304), (1280, 11008)])
def test_fp8_shapes(ffn, oracle_lib, d, ffn_):
    """One k-block, odd numbers of k-blocks and of 64-row groups, one split."""
    inp = synth.make_fp8_inputs(synth.C6_DECODE_FP8, seed=d, rows=4, d=d, ffn=ffn_)
    assert_lowp(to_host64(run_fp8(ffn, inp)), oracle_lib.fp8_block_from_inputs(inp))


def _finite_codes(lo_exp: int, hi_exp: int) -> np.ndarray:
    """Every finite e4m3 code (both signs) whose exponent field is in [lo_exp, hi_exp]."""
    out = []
    for b in range(256):
        e, f = (b >> 3) & 15, b & 7
        if lo_exp <= e <= hi_exp and not (e == 15 and f == 7):
            out.append(b)
    return np.array(out, dtype=np.uint8)


@pytest.mark.parametrize("cls,lo,hi", [("subnormal", 0, 0), ("small", 1, 4), ("middle", 5, 10),
                                        ("large", 11, 15), ("all", 0, 15)])
def test_fp8_code_classes(ffn, oracle_lib, cls, lo, hi):
    """W_down drawn from one class of codes only, so a decoding error in that
    class is not hidden behind larger values: every code of the class occurs
    many times."""
    inp = synth.make_fp8_inputs(synth.C6_DECODE_FP8, seed=11, rows=8, d=512, ffn=1024)
    codes = _finite_codes(lo, hi)
    rng = np.random.default_rng(lo * 16 + hi)
    inp["c_down"] = codes[rng.integers(0, codes.size, size=inp["c_down"].shape)].astype(np.uint8)
    assert_lowp(to_host64(run_fp8(ffn, inp)), oracle_lib.fp8_block_from_inputs(inp))


def test_fp8_single_code_probe(ffn, oracle_lib):
    """Gate and up all zero but for two codes each: the output isolates those
    codes' positions, values and row scales through the whole path."""
    inp = synth.make_fp8_inputs(synth.C6_DECODE_FP8, seed=2, rows=2, d=256, ffn=256)
    for name in ("gate", "up"):
        c = np.zeros((256, 256), dtype=np.uint8)
        c[37, 161] = 0xD3   # -2^(10-7) * 1.375 = -11
        c[37, 5] = 0x3A     # 2^(7-7) * 1.25 = 1.25
        c[200, 255] = 0x05  # subnormal 5 * 2^-9
        inp["c_" + name] = c
    y = to_host64(run_fp8(ffn, inp))
    assert_lowp(y, oracle_lib.fp8_block_from_inputs(inp))


def test_fp8_residual(ffn, oracle_lib):
    inp = synth.make_fp8_inputs(synth.C6_DECODE_FP8, seed=4, rows=5, d=1024, ffn=2048)
    y = run_fp8(ffn, inp, flags=ffn.FFN_RESIDUAL)
    assert_lowp(to_host64(y), oracle_lib.fp8_block_from_inputs(inp, residual=True))


def test_fp8_zero_scales_give_zero(ffn):
    """Row scales of zero on W_down: y is exactly zero (and x with the skip
    connection), whatever the codes."""
    import torch
    inp = synth.make_fp8_inputs(synth.C6_DECODE_FP8, seed=6, rows=3, d=256, ffn=512)
    inp["s_down"] = np.zeros_like(inp["s_down"])
    y = run_fp8(ffn, inp)
    assert torch.count_nonzero(y.float()).item() == 0
    y = run_fp8(ffn, inp, flags=ffn.FFN_RESIDUAL)
    assert torch.equal(y.view(torch.int16).cpu(), torch.from_numpy(inp["x"].view(np.int16)))


def test_fp8_deterministic(ffn):
    import hashlib

    import torch
    inp = synth.make_fp8_inputs(synth.C6_DECODE_FP8, seed=5, rows=8, d=1024, ffn=2048)
    hs = {hashlib.sha256(run_fp8(ffn, inp).view(torch.int16).cpu().numpy().tobytes()).hexdigest()
          for _ in range(3)}
    assert len(hs) == 1


def test_fp8_rejects_float8_dtype_mismatch(ffn):
    import torch
    inp = synth.make_fp8_inputs(synth.C6_DECODE_FP8, seed=3, rows=2, d=256, ffn=256)
    c, s = fp8_dev(inp, "gate")
    with pytest.raises(TypeError):
        ffn.ffn_block_forward_fp8(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"), (c, s.double()),
                                  fp8_dev(inp, "up"), fp8_dev(inp, "down"), eps=1e-5)
    # torch's own e4m3 dtype is accepted as the codes
    y = ffn.ffn_block_forward_fp8(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"),
                                  (c.view(torch.float8_e4m3fn), s), fp8_dev(inp, "up"), fp8_dev(inp, "down"),
                                  eps=inp["cfg"].eps)
    assert torch.equal(y, run_fp8(ffn, inp))
