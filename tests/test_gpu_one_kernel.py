"""FFN_DECODE_ONE_KERNEL: the decode block as one persistent kernel
("Megakernels on Mac: What Fusion Saves and What It Costs", "Dependencies and
synchronization"), against the float64 oracle on every weight format, with
the skip connection and the handed-on row statistics, call after call on one
stream (epoch-stamped flags), and on two streams at once (one control block
each).  The default three-kernel chain computes the same fragments and
partial sums in the same orders, so the two agree within the bound of each
other."""

import hashlib

import numpy as np
import pytest

import synth
from gpu_util import assert_lowp, fp8_dev, q4_dev, q8_dev, to_dev, to_host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ffn():
    from transformer_ffn_rmsnorm_gb300 import ffn as m
    return m


def dev_args(inp):
    return [to_dev(inp[k], "bf16") for k in ("x", "g", "w_gate", "w_up", "w_down")]


@pytest.mark.parametrize("rows,d,ffn_", [(1, 1024, 2816), (5, 520, 648), (8, 1024, 2816), (13, 512, 1536),
                                         (16, 2048, 5632), (33, 1024, 2816), (64, 512, 1024)])
def test_one_kernel_bf16(ffn, oracle_lib, rows, d, ffn_):
    """bf16 weights (hi + lo operands), one to eight token tiles, d and ffn
    multiples of 8 only (ragged TMA boxes at both ends)."""
    inp = synth.make_block_inputs(synth.C3_DECODE_BF16, seed=500 + rows, rows=rows, d=d, ffn=ffn_)
    args = dev_args(inp)
    flags = ffn.FFN_DECODE_ONE_KERNEL | (ffn.FFN_PATH_GEMV if rows > 16 else 0)
    y = ffn.ffn_block_forward(*args, eps=inp["cfg"].eps, flags=flags)
    assert_lowp(to_host64(y), oracle_lib.block_from_inputs(inp))
    ffn.ffn_device_status()


@pytest.mark.parametrize("residual", [False, True])
def test_one_kernel_prepared(ffn, oracle_lib, residual):
    inp = synth.make_block_inputs(synth.C3_DECODE_BF16, seed=77, rows=8, d=1024, ffn=2816)
    args = dev_args(inp)
    args[2:] = [ffn.ffn_prepare_weights(w) for w in args[2:]]
    flags = ffn.FFN_DECODE_ONE_KERNEL | ffn.FFN_PREPARED_WEIGHTS | (ffn.FFN_RESIDUAL if residual else 0)
    y = ffn.ffn_block_forward(*args, eps=inp["cfg"].eps, flags=flags)
    assert_lowp(to_host64(y), oracle_lib.block_from_inputs(inp, residual=residual))


@pytest.mark.parametrize("rows", [3, 8, 16])
def test_one_kernel_q4(ffn, oracle_lib, rows):
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=rows, rows=rows, d=1024, ffn=2816)
    cfg = inp["cfg"]
    y = ffn.ffn_block_forward_q4(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"), q4_dev(inp, "gate"),
                                 q4_dev(inp, "up"), q4_dev(inp, "down"), ffn=cfg.ffn, eps=cfg.eps,
                                 flags=ffn.FFN_DECODE_ONE_KERNEL)
    assert_lowp(to_host64(y), oracle_lib.q4_block_from_inputs(inp))


def test_one_kernel_q4_full_size(ffn, oracle_lib):
    """8 x 5120 -> 17408: d above the 4096 values a norm CTA holds in
    registers (the two-pass norm)."""
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=0)
    cfg = inp["cfg"]
    y = ffn.ffn_block_forward_q4(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"), q4_dev(inp, "gate"),
                                 q4_dev(inp, "up"), q4_dev(inp, "down"), ffn=cfg.ffn, eps=cfg.eps,
                                 flags=ffn.FFN_DECODE_ONE_KERNEL)
    assert_lowp(to_host64(y), oracle_lib.q4_block_from_inputs(inp))


@pytest.mark.parametrize("residual", [False, True])
def test_one_kernel_fp8_q8(ffn, oracle_lib, residual):
    R = ffn.FFN_RESIDUAL if residual else 0
    inp = synth.make_fp8_inputs(synth.C6_DECODE_FP8, seed=21, rows=7, d=1024, ffn=2048)
    y = ffn.ffn_block_forward_fp8(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"), fp8_dev(inp, "gate"),
                                  fp8_dev(inp, "up"), fp8_dev(inp, "down"), eps=inp["cfg"].eps,
                                  flags=ffn.FFN_DECODE_ONE_KERNEL | R)
    assert_lowp(to_host64(y), oracle_lib.fp8_block_from_inputs(inp, residual=residual))
    inp = synth.make_q8_inputs(synth.C7_DECODE_Q8, seed=22, rows=7, d=1024, ffn=2048)
    y = ffn.ffn_block_forward_q8(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"), q8_dev(inp, "gate"),
                                 q8_dev(inp, "up"), q8_dev(inp, "down"), eps=inp["cfg"].eps,
                                 flags=ffn.FFN_DECODE_ONE_KERNEL | R)
    assert_lowp(to_host64(y), oracle_lib.q8_block_from_inputs(inp, residual=residual))


def test_one_kernel_chained_statistics(ffn, oracle_lib):
    """Two chained blocks, the one-kernel form: y_sumsq of block 1 is the sum
    of squares of its stored y, and block 2 on it matches block 2 reducing
    its rows itself (default path) within the bound."""
    import torch
    cfg = synth.C3_DECODE_BF16
    a1 = dev_args(synth.make_block_inputs(cfg, seed=31, rows=8, d=1024, ffn=2816))
    a2 = dev_args(synth.make_block_inputs(cfg, seed=32, rows=8, d=1024, ffn=2816))
    F = ffn.FFN_DECODE_ONE_KERNEL | ffn.FFN_RESIDUAL
    y1, ss1 = ffn.ffn_block_forward_chained(*a1, eps=cfg.eps, flags=F)
    y2, ss2 = ffn.ffn_block_forward_chained(y1, *a2[1:], eps=cfg.eps, flags=F, x_sumsq=ss1)
    ref = ffn.ffn_block_forward(y1, *a2[1:], eps=cfg.eps, flags=ffn.FFN_RESIDUAL)
    torch.cuda.synchronize()
    v1 = to_host64(y1)
    assert np.allclose(ss1.cpu().numpy(), np.sum(v1 * v1, axis=1), rtol=1e-5, atol=0)
    a, b = to_host64(y2), to_host64(ref)
    assert np.abs(a - b).max() <= 2e-2 * np.sqrt(np.mean(b * b))
    ffn.ffn_device_status()


def test_one_kernel_many_calls_and_determinism(ffn, oracle_lib):
    """Thirty calls in a row on one stream and workspace, alternating with
    the default chain: every one-kernel call bitwise equal to the first (the
    control block's flags carry each call's epoch), results in bound."""
    import torch
    inp = synth.make_block_inputs(synth.C3_DECODE_BF16, seed=40, rows=8, d=1024, ffn=2816)
    args = dev_args(inp)
    ws = ffn.workspace(ffn.ffn_block_workspace_bytes(8, 1024, 2816, torch.bfloat16, 0), args[0].device)
    outs = []
    for i in range(30):
        y = ffn.ffn_block_forward(*args, eps=inp["cfg"].eps, flags=ffn.FFN_DECODE_ONE_KERNEL, ws=ws)
        outs.append(y)
        if i % 3 == 0:
            ffn.ffn_block_forward(*args, eps=inp["cfg"].eps, ws=ws)
    torch.cuda.synchronize()
    h = {hashlib.sha256(y.view(torch.int16).cpu().numpy().tobytes()).hexdigest() for y in outs}
    assert len(h) == 1
    assert_lowp(to_host64(outs[-1]), oracle_lib.block_from_inputs(inp))
    ffn.ffn_device_status()


def test_one_kernel_two_streams(ffn, oracle_lib):
    """Calls on two streams at once, each with its own workspace: each stream
    has its own control block, so neither sees the other's flags."""
    import torch
    inps = [synth.make_block_inputs(synth.C3_DECODE_BF16, seed=50 + i, rows=8, d=1024, ffn=2816)
            for i in range(2)]
    argss = [dev_args(inp) for inp in inps]
    streams = [torch.cuda.Stream() for _ in range(2)]
    torch.cuda.synchronize()
    outs = [[], []]
    for _ in range(10):
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                outs[i].append(ffn.ffn_block_forward(*argss[i], eps=inps[i]["cfg"].eps,
                                                     flags=ffn.FFN_DECODE_ONE_KERNEL))
    torch.cuda.synchronize()
    for i in range(2):
        ref = oracle_lib.block_from_inputs(inps[i])
        for y in (outs[i][0], outs[i][-1]):
            assert_lowp(to_host64(y), ref)
    ffn.ffn_device_status()
