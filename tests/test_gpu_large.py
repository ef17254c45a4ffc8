"""Large shapes: a 70B-class layer (d 8192, ffn 28672) through the decode
kernels in every weight format and through the prefill GEMMs, and prefill
batches whose intermediate tensors pass 2^31 bytes (every index and offset
must be 64-bit).  The oracle runs on all rows for decode and on sampled rows
(rows are independent) for prefill."""

import numpy as np
import pytest

import synth
from gpu_util import assert_lowp, fp8_dev, q4_dev, q8_dev, to_dev, to_host64

pytestmark = pytest.mark.gpu

D70, F70 = 8192, 28672


@pytest.fixture(scope="module")
def ffn():
    from transformer_ffn_rmsnorm_gb300 import ffn as m
    return m


def block_args(inp):
    return [to_dev(inp[k], "bf16") for k in ("x", "g", "w_gate", "w_up", "w_down")]


def test_decode_70b_bf16(ffn, oracle_lib):
    inp = synth.make_block_inputs(synth.C3_DECODE_BF16, seed=70, rows=8, d=D70, ffn=F70)
    y = ffn.ffn_block_forward(*block_args(inp), eps=inp["cfg"].eps)
    assert_lowp(to_host64(y), oracle_lib.block_from_inputs(inp))


def test_decode_70b_fp8(ffn, oracle_lib):
    inp = synth.make_fp8_inputs(synth.C6_DECODE_FP8, seed=71, rows=12, d=D70, ffn=F70)
    y = ffn.ffn_block_forward_fp8(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"), fp8_dev(inp, "gate"),
                                  fp8_dev(inp, "up"), fp8_dev(inp, "down"), eps=inp["cfg"].eps)
    assert_lowp(to_host64(y), oracle_lib.fp8_block_from_inputs(inp))


def test_decode_70b_q8(ffn, oracle_lib):
    inp = synth.make_q8_inputs(synth.C7_DECODE_Q8, seed=72, rows=8, d=D70, ffn=F70)
    y = ffn.ffn_block_forward_q8(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"), q8_dev(inp, "gate"),
                                 q8_dev(inp, "up"), q8_dev(inp, "down"), eps=inp["cfg"].eps)
    assert_lowp(to_host64(y), oracle_lib.q8_block_from_inputs(inp))


def test_decode_70b_q4(ffn, oracle_lib):
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=73, rows=8, d=D70, ffn=F70)
    y = ffn.ffn_block_forward_q4(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"), q4_dev(inp, "gate"),
                                 q4_dev(inp, "up"), q4_dev(inp, "down"), ffn=F70, eps=inp["cfg"].eps)
    assert_lowp(to_host64(y), oracle_lib.q4_block_from_inputs(inp))


def test_prefill_70b_prepared_sampled(ffn, oracle_lib):
    rows = 1024
    inp = synth.make_block_inputs(synth.C4_PREFILL_BF16, seed=74, rows=rows, d=D70, ffn=F70)
    args = block_args(inp)
    args[2:] = [ffn.ffn_prepare_weights(w) for w in args[2:]]
    y = to_host64(ffn.ffn_block_forward(*args, eps=inp["cfg"].eps, flags=ffn.FFN_PREPARED_WEIGHTS))
    sel = np.r_[0:6, 509:515, rows - 6:rows]
    assert_lowp(y[sel], oracle_lib.block_from_inputs(inp, rows=sel))


@pytest.mark.parametrize("rows,ffn_,flags", [(16384, 32768, 2), (32768, 32768, 64)])
def test_prefill_tensors_past_2_gib(ffn, oracle_lib, rows, ffn_, flags):
    """Unfused (flags 2): fp32 G and U of 16384 x 32768 (2.1 GB each).
    Prepared fused (flags 64): h of 32768 x 32768 fp16 (2.1 GB).  Rows
    sampled at the start, the middle and the end of the batch."""
    inp = synth.make_block_inputs(synth.C4_PREFILL_BF16, seed=rows, rows=rows, d=1024, ffn=ffn_)
    args = block_args(inp)
    if flags & ffn.FFN_PREPARED_WEIGHTS:
        args[2:] = [ffn.ffn_prepare_weights(w) for w in args[2:]]
    y = ffn.ffn_block_forward(*args, eps=inp["cfg"].eps, flags=flags)
    import torch
    sel = np.r_[0:4, rows // 2 - 2:rows // 2 + 2, rows - 4:rows]
    got = to_host64(y[torch.from_numpy(sel).to(y.device)])
    assert_lowp(got, oracle_lib.block_from_inputs(inp, rows=sel))
    ffn.ffn_device_status()
