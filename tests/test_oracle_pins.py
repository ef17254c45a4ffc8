"""The oracle against what the mathematics fixes (CPU only)."""

import math

import numpy as np
import pytest

import oracle_pins
import synth
from oracle import widen


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(oracle_lib, pin):
    pin(oracle_lib)


def test_numpy_statement_cross_check(oracle_lib):
    """An independent matrix statement of the block in numpy float64."""
    inp = synth.make_block_inputs(synth.C1_TINY_F32, seed=3, rows=9, d=64, ffn=96)
    x, g = widen(inp["x"], "f32"), widen(inp["g"], "f32")
    wg, wu, wd = (widen(inp[k], "f32") for k in ("w_gate", "w_up", "w_down"))
    eps = inp["cfg"].eps
    n = x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + eps) * g
    G, U = n @ wg.T, n @ wu.T
    y = (G / (1.0 + np.exp(-G)) * U) @ wd.T
    got = oracle_lib.block_from_inputs(inp)
    assert np.allclose(got, y, rtol=1e-12, atol=1e-13)


def test_thread_count_does_not_change_bits(oracle_lib):
    inp = synth.make_block_inputs(synth.C3_DECODE_BF16, seed=1, rows=3, d=128, ffn=256)
    a = oracle_lib.block_from_inputs(inp, nthreads=1)
    b = oracle_lib.block_from_inputs(inp, nthreads=5)
    assert np.array_equal(a, b)


def test_widen_is_exact():
    rng = np.random.default_rng(0)
    v = rng.standard_normal(1000)
    b = synth.round_to_storage(v, "bf16")
    w = widen(b, "bf16")
    # bfloat16 keeps 8 significant bits: the value re-rounds to itself
    assert np.array_equal(synth.round_to_storage(w, "bf16"), b)
    assert np.all(np.abs(w - v) <= np.abs(v) * 2.0 ** -8)
    h = synth.round_to_storage(v, "f16")
    assert np.array_equal(widen(h, "f16"), h.astype(np.float64))


def test_q4_block_uses_dequantised_weights(oracle_lib):
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=2, rows=2, d=128, ffn=256)
    wg = inp["q_gate"].astype(np.float64) * np.repeat(inp["s_gate"].astype(np.float64), 32, axis=1)
    wu = inp["q_up"].astype(np.float64) * np.repeat(inp["s_up"].astype(np.float64), 32, axis=1)
    wd = inp["q_down"].astype(np.float64) * np.repeat(inp["s_down"].astype(np.float64), 32, axis=1)
    y_ref = oracle_lib.ffn_block(widen(inp["x"], "bf16"), widen(inp["g"], "bf16"), wg, wu, wd,
                                 inp["cfg"].eps)
    assert np.array_equal(oracle_lib.q4_block_from_inputs(inp), y_ref)
    assert math.isfinite(float(np.abs(y_ref).max()))
