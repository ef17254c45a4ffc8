"""ffn_block_forward_q8 (Q8_0 weights) on the GPU against the oracle, which
dequantises the int8 codes and fp16 block scales itself (float64); and the
Q8_0 weights prepared for the tensor-core path."""

import numpy as np
import pytest

import synth
from gpu_util import assert_lowp, q8_dev, to_dev, to_host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ffn():
    from transformer_ffn_rmsnorm_gb300 import ffn as m
    return m


def run_q8(ffn, inp, flags=0):
    return ffn.ffn_block_forward_q8(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"), q8_dev(inp, "gate"),
                                    q8_dev(inp, "up"), q8_dev(inp, "down"), eps=inp["cfg"].eps, flags=flags)


def test_q8_full_size(ffn, oracle_lib):
    """8 rows, d=4096, ffn=14336."""
    inp = synth.make_q8_inputs(synth.C7_DECODE_Q8, seed=0)
    assert_lowp(to_host64(run_q8(ffn, inp)), oracle_lib.q8_block_from_inputs(inp))


@pytest.mark.parametrize("rows", [1, 3, 8, 9, 16, 20, 33])
def test_q8_rows(ffn, oracle_lib, rows):
    inp = synth.make_q8_inputs(synth.C7_DECODE_Q8, seed=rows, rows=rows, d=1024, ffn=2816)
    assert_lowp(to_host64(run_q8(ffn, inp)), oracle_lib.q8_block_from_inputs(inp))


@pytest.mark.parametrize("d,ffn_", [(256, 256), (768, 1280), (4096, 2304), (1280, 11008 + 256)])
def test_q8_shapes(ffn, oracle_lib, d, ffn_):
    """One k-block, odd numbers of k-blocks and of 64-row groups."""
    inp = synth.make_q8_inputs(synth.C7_DECODE_Q8, seed=d, rows=4, d=d, ffn=ffn_)
    assert_lowp(to_host64(run_q8(ffn, inp)), oracle_lib.q8_block_from_inputs(inp))


def test_q8_extreme_codes_and_scales(ffn, oracle_lib):
    """Codes at -128 and 127 and mixed-sign block scales in every matrix."""
    inp = synth.make_q8_inputs(synth.C7_DECODE_Q8, seed=12, rows=8, d=512, ffn=1024)
    rng = np.random.default_rng(5)
    for name in ("gate", "up", "down"):
        q = inp["q8_" + name]
        q[rng.random(q.shape) < 0.25] = -128
        q[rng.random(q.shape) < 0.25] = 127
        s = inp["q8s_" + name].view(np.float16).copy()
        s *= rng.choice(np.array([-1, 1], dtype=np.float16), s.shape)
        inp["q8s_" + name] = s.view(np.uint16)
    assert_lowp(to_host64(run_q8(ffn, inp)), oracle_lib.q8_block_from_inputs(inp))


def test_q8_single_code_probe(ffn, oracle_lib):
    """Gate and up zero but for a few codes: position, sign, block scale."""
    inp = synth.make_q8_inputs(synth.C7_DECODE_Q8, seed=2, rows=2, d=256, ffn=256)
    for name in ("gate", "up"):
        q = np.zeros((256, 256), dtype=np.int8)
        q[37, 161], q[37, 5], q[200, 255] = -100, 77, 1
        inp["q8_" + name] = q
    assert_lowp(to_host64(run_q8(ffn, inp)), oracle_lib.q8_block_from_inputs(inp))


def test_q8_residual(ffn, oracle_lib):
    inp = synth.make_q8_inputs(synth.C7_DECODE_Q8, seed=4, rows=5, d=1024, ffn=2048)
    assert_lowp(to_host64(run_q8(ffn, inp, ffn.FFN_RESIDUAL)), oracle_lib.q8_block_from_inputs(inp, residual=True))


def test_q8_deterministic(ffn):
    import hashlib

    import torch
    inp = synth.make_q8_inputs(synth.C7_DECODE_Q8, seed=5, rows=8, d=1024, ffn=2048)
    hs = {hashlib.sha256(run_q8(ffn, inp).view(torch.int16).cpu().numpy().tobytes()).hexdigest() for _ in range(3)}
    assert len(hs) == 1


def test_prepare_q8_bit_exact(ffn, oracle_lib):
    import torch
    inp = synth.make_q8_inputs(synth.C7_DECODE_Q8, seed=9, rows=2, d=512, ffn=768)
    got = ffn.ffn_prepare_weights_q8(q8_dev(inp, "gate"))
    w = oracle_lib.q8_dequant(inp["q8_gate"], inp["q8s_gate"], 768, 512)
    assert np.array_equal(got.view(torch.int16).cpu().numpy().view(np.uint16),
                          (w * 256.0).astype(np.float16).view(np.uint16))
    ffn.ffn_device_status()


@pytest.mark.parametrize("rows,d,ffn_", [(40, 256, 512), (700, 1024, 1536)])
def test_prefill_from_q8_weights(ffn, oracle_lib, rows, d, ffn_):
    inp = synth.make_q8_inputs(synth.C7_DECODE_Q8, seed=rows, rows=rows, d=d, ffn=ffn_)
    w = [ffn.ffn_prepare_weights_q8(q8_dev(inp, n)) for n in ("gate", "up", "down")]
    y = to_host64(ffn.ffn_block_forward(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"), *w,
                                        eps=inp["cfg"].eps, flags=ffn.FFN_PREPARED_WEIGHTS))
    sel = np.r_[0:20, rows - 20:rows]
    assert_lowp(y[sel], oracle_lib.q8_block_from_inputs(inp, rows=sel))
