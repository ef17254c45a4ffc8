"""FFN_RESIDUAL: y = x + W_down(silu(W_gate n) * (W_up n)), x added before y's
one rounding, on every path, against the oracle's float64 skip connection."""

import numpy as np
import pytest

import synth
from gpu_util import assert_f32, assert_lowp, q4_dev, to_dev, to_host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ffn():
    from transformer_ffn_rmsnorm_gb300 import ffn as m
    return m


def block(ffn, inp, flags):
    dt = inp["cfg"].dtype
    args = [to_dev(inp[k], dt) for k in ("x", "g", "w_gate", "w_up", "w_down")]
    if flags & ffn.FFN_PREPARED_WEIGHTS:
        args[2:] = [ffn.ffn_prepare_weights(w) for w in args[2:]]
    return ffn.ffn_block_forward(*args, eps=inp["cfg"].eps, flags=flags | ffn.FFN_RESIDUAL)


def test_residual_fp32_simt(ffn, oracle_lib):
    inp = synth.make_block_inputs(synth.C1_TINY_F32, seed=3)
    assert_f32(to_host64(block(ffn, inp, 0)), oracle_lib.block_from_inputs(inp, residual=True))


@pytest.mark.parametrize("rows", [1, 8, 13])
@pytest.mark.parametrize("dtype,flags", [("bf16", 0), ("f16", 0), ("bf16", 64)])
def test_residual_decode(ffn, oracle_lib, rows, dtype, flags):
    cfg = synth.BlockConfig("t", rows, 1024, 2816, 1e-5, dtype)
    inp = synth.make_block_inputs(cfg, seed=300 + rows)
    assert_lowp(to_host64(block(ffn, inp, flags)), oracle_lib.block_from_inputs(inp, residual=True))


@pytest.mark.parametrize("flags", [0, 2, 64])
@pytest.mark.parametrize("rows,d,ffn_", [(300, 512, 704), (2048, 4096, 1280)])
def test_residual_prefill(ffn, oracle_lib, flags, rows, d, ffn_):
    cfg = synth.BlockConfig("t", rows, d, ffn_, 1e-6, "bf16")
    inp = synth.make_block_inputs(cfg, seed=rows + 7)
    y = to_host64(block(ffn, inp, flags))
    sel = np.unique(np.concatenate([np.arange(0, rows, 37), [rows - 1]]))
    assert_lowp(y[sel], oracle_lib.block_from_inputs(inp, rows=sel, residual=True))


@pytest.mark.parametrize("rows", [8, 300])
def test_residual_zero_down_returns_x(ffn, rows):
    """W_down = 0: the projection is exactly zero, so y == x bit for bit."""
    import torch
    cfg = synth.BlockConfig("t", rows, 512, 704, 1e-6, "bf16")
    inp = synth.make_block_inputs(cfg, seed=21)
    inp["w_down"] = np.zeros_like(inp["w_down"])
    x = to_dev(inp["x"], "bf16")
    y = block(ffn, inp, 0)
    assert torch.equal(y.view(torch.int16), x.view(torch.int16))


def test_residual_q4(ffn, oracle_lib):
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=5, rows=9, d=1024, ffn=2816)
    cfg = inp["cfg"]
    y = ffn.ffn_block_forward_q4(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"), q4_dev(inp, "gate"),
                                 q4_dev(inp, "up"), q4_dev(inp, "down"), ffn=cfg.ffn, eps=cfg.eps,
                                 flags=ffn.FFN_RESIDUAL)
    assert_lowp(to_host64(y), oracle_lib.q4_block_from_inputs(inp, residual=True))


def test_residual_host_entry(ffn, oracle_lib):
    """Through ffn_block_forward_host (three chunks): the same bytes as the
    device-buffer call."""
    import torch
    inp = synth.make_block_inputs(synth.C4_PREFILL_BF16, seed=2, rows=3500, d=256, ffn=384)
    g, wg, wu, wd = (to_dev(inp[k], "bf16") for k in ("g", "w_gate", "w_up", "w_down"))
    xh = torch.from_numpy(np.ascontiguousarray(inp["x"]).view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = ffn.ffn_block_forward_host(xh, g, wg, wu, wd, eps=1e-6, flags=ffn.FFN_RESIDUAL)
    torch.cuda.current_stream().synchronize()
    yd = ffn.ffn_block_forward(to_dev(inp["x"], "bf16"), g, wg, wu, wd, eps=1e-6, flags=ffn.FFN_RESIDUAL)
    assert torch.equal(yh.view(torch.int16), yd.cpu().view(torch.int16))
    sel = np.r_[0:20, 3480:3500]
    assert_lowp(to_host64(yh)[sel], oracle_lib.block_from_inputs(inp, rows=sel, residual=True))
