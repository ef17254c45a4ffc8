"""The oracle reproduces its stored regression anchors (CPU only).

The anchors were written by tests/golden/make_golden.py; across machines libm's
exp may differ in the last bit, hence the 1e-13 relative bound."""
import os

import numpy as np

import synth

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    return np.loadtxt(os.path.join(HERE, name), comments="#")


def test_block_tiny_f32(oracle_lib):
    inp = synth.make_block_inputs(synth.C1_TINY_F32, seed=0, rows=4, d=32, ffn=48)
    y = oracle_lib.block_from_inputs(inp)
    assert np.allclose(y, _load("block_tiny_f32_seed0_4x32x48.txt"), rtol=1e-13, atol=1e-15)


def test_block_q4(oracle_lib):
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=0, rows=2, d=128, ffn=256)
    y = oracle_lib.q4_block_from_inputs(inp)
    assert np.allclose(y, _load("block_q4_seed0_2x128x256.txt"), rtol=1e-13, atol=1e-15)
