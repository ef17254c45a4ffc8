"""Quantised weights prepared for the tensor-core path: ffn_prepare_weights_fp8
and ffn_prepare_weights_q4 against the oracle's own dequantisation (fp16 of
w * 2^8, one correct rounding), then whole prefill blocks on the prepared
weights against the oracle on the exact quantised weights."""

import numpy as np
import pytest

import synth
from gpu_util import assert_lowp, fp8_dev, q4_dev, to_dev, to_host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ffn():
    from transformer_ffn_rmsnorm_gb300 import ffn as m
    return m


def f16_bits(a64: np.ndarray) -> np.ndarray:
    """fp16 bit patterns of float64 values, round to nearest even (numpy)."""
    return a64.astype(np.float16).view(np.uint16)


def test_prepare_fp8_bit_exact(ffn, oracle_lib):
    """Every finite code, scales spanning normal and subnormal fp16 results."""
    import torch
    rng = np.random.default_rng(21)
    out, inn = 96, 512
    finite = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], dtype=np.uint8)
    codes = finite[rng.integers(0, finite.size, (out, inn))]
    scales = (np.exp(rng.uniform(np.log(1e-6), np.log(0.5), out)) * rng.choice([-1, 1], out)).astype(np.float32)
    got = ffn.ffn_prepare_weights_fp8((torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda()))
    w = oracle_lib.fp8_dequant(codes, scales, out, inn)
    assert np.array_equal(got.view(torch.int16).cpu().numpy().view(np.uint16), f16_bits(w * 256.0))
    ffn.ffn_device_status()


@pytest.mark.parametrize("d,ffn_", [(1024, 640), (96, 160), (416, 224)])
def test_prepare_q4_bit_exact(ffn, oracle_lib, d, ffn_):
    """Whole 128-weight groups and rows ending in a partial group (1 and 3
    blocks): every weight written once, nothing past the row."""
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=4, rows=2, d=d, ffn=ffn_)
    qs, sc = q4_dev(inp, "gate")
    got = ffn.ffn_prepare_weights_q4((qs, sc), d)
    w = oracle_lib.q4_dequant(inp["qs_gate"], inp["sc_gate"], ffn_, d)
    import torch
    assert got.shape == (ffn_, d)
    assert np.array_equal(got.view(torch.int16).cpu().numpy().view(np.uint16), f16_bits(w * 256.0))
    ffn.ffn_device_status()


def test_prepare_fp8_range(ffn):
    """|w| * 2^8 beyond fp16's range: infinite, and FFN_ERR_RANGE recorded."""
    import torch
    codes = np.full((1, 16), 0x38, dtype=np.uint8)   # e4m3 1.0
    codes[0, 3] = 0x7E                                # 448
    scales = np.array([1.0], dtype=np.float32)
    got = ffn.ffn_prepare_weights_fp8((torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda()))
    with pytest.raises(ffn.FFNError) as e:
        ffn.ffn_device_status()
    assert e.value.status == 10
    assert torch.isinf(got[0, 3]).item() and got[0, 0].item() == 256.0


def prefill_fp8(ffn, inp, flags=0):
    P = ffn.FFN_PREPARED_WEIGHTS
    w = [ffn.ffn_prepare_weights_fp8(fp8_dev(inp, n)) for n in ("gate", "up", "down")]
    return ffn.ffn_block_forward(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"), *w, eps=inp["cfg"].eps,
                                 flags=P | flags)


@pytest.mark.parametrize("rows,d,ffn_", [(40, 256, 384), (300, 512, 1024), (1030, 1024, 2816)])
def test_prefill_from_fp8_weights(ffn, oracle_lib, rows, d, ffn_):
    """Through the tensor-core GEMMs (rows > 16; CTA pairs from 256 rows)."""
    inp = synth.make_fp8_inputs(synth.C6_DECODE_FP8, seed=rows, rows=rows, d=d, ffn=ffn_)
    y = to_host64(prefill_fp8(ffn, inp))
    sel = np.r_[0:20, rows - 20:rows] if rows > 64 else np.arange(rows)
    assert_lowp(y[sel], oracle_lib.fp8_block_from_inputs(inp, rows=sel))


def test_prefill_from_fp8_weights_residual(ffn, oracle_lib):
    inp = synth.make_fp8_inputs(synth.C6_DECODE_FP8, seed=5, rows=200, d=256, ffn=512)
    y = to_host64(prefill_fp8(ffn, inp, ffn.FFN_RESIDUAL))
    assert_lowp(y, oracle_lib.fp8_block_from_inputs(inp, residual=True))


@pytest.mark.parametrize("rows,d,ffn_", [(40, 256, 384), (600, 1024, 1536)])
def test_prefill_from_q4_weights(ffn, oracle_lib, rows, d, ffn_):
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=rows, rows=rows, d=d, ffn=ffn_)
    P = ffn.FFN_PREPARED_WEIGHTS
    w = [ffn.ffn_prepare_weights_q4(q4_dev(inp, n), i) for n, i in (("gate", d), ("up", d), ("down", ffn_))]
    y = to_host64(ffn.ffn_block_forward(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"), *w,
                                        eps=inp["cfg"].eps, flags=P))
    sel = np.r_[0:20, rows - 20:rows]
    assert_lowp(y[sel], oracle_lib.q4_block_from_inputs(inp, rows=sel))
