"""ffn_block_forward_chained: the RMSNorm reduction handed from one block to
the next ("Megakernels on Mac: What Fusion Saves and What It Costs",
"Dependencies and synchronization").

y_sumsq, the rows' sums of squares of the stored y, is checked on every path
(decode kernels, tensor-core GEMMs with and without a split reduction, fp32)
  * against the float64 oracle's statistic of its own y: with |y - y_o| <=
    2e-2 * rms(y_o) element by element (the block's bound), a row's sum of
    squares can move by at most 2e-2 * rms * (2 * sum_c |y_o| + d * 2e-2 *
    rms) -- the test's bound;
  * as a property of the call: it is the sum of squares of the y the call
    returned (fp32 accumulation, relative 1e-5).
x_sumsq is checked by running the block on the oracle's own statistic of x
(exact, in float64, rounded once to fp32) against the oracle's block, and a
two-block chain (the first call's y and y_sumsq feeding the second) against
the second block run with its own reduction.  y itself is bitwise the same
as ffn_block_forward's."""

import numpy as np
import pytest

import synth
from gpu_util import BF16_MAX, assert_dtype, to_dev, to_host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ffn():
    from transformer_ffn_rmsnorm_gb300 import ffn as m
    return m


def dev(inp, dtype):
    import torch
    names = ("x", "g", "w_gate", "w_up", "w_down")
    if dtype == "bf16":
        return [to_dev(inp[k], "bf16") for k in names]
    return [torch.from_numpy(np.ascontiguousarray(inp[k])).cuda() for k in names]


def check_sumsq(ss_gpu, y_gpu64, y_ref, max_rel):
    """ss_gpu against the oracle's statistic of its own y (bound from the
    block's max bound) and against the returned y (property)."""
    rms = float(np.sqrt(np.mean(y_ref * y_ref)))
    d = y_ref.shape[1]
    ss_ref = np.sum(y_ref * y_ref, axis=1)
    tol = max_rel * rms * (2.0 * np.sum(np.abs(y_ref), axis=1) + d * max_rel * rms)
    err = np.abs(ss_gpu - ss_ref)
    assert np.all(err <= tol), f"worst row: err {err.max():.4e} vs bound {tol[np.argmax(err - tol)]:.4e}"
    own = np.sum(y_gpu64 * y_gpu64, axis=1)
    assert np.allclose(ss_gpu, own, rtol=1e-5, atol=0), np.max(np.abs(ss_gpu - own) / own)


CASES = [
    # (label, config, rows, d, ffn, flags)
    ("decode_stream", synth.C3_DECODE_BF16, 8, 1024, 2816, 0),
    ("decode_two_tiles", synth.C3_DECODE_BF16, 13, 512, 1536, 0),
    ("decode_ragged", synth.C3_DECODE_BF16, 5, 520, 648, 0),        # d, ffn not multiples of 64
    ("gemm_split_reduce", synth.C4_PREFILL_BF16, 200, 1024, 2816, 0),
    ("gemm_tiles", synth.C4_PREFILL_BF16, 2500, 1024, 768, 0),      # unsplit, ragged last row block
    ("gemm_prepared", synth.C4_PREFILL_BF16, 2500, 1024, 768, 64),
    ("fp32", synth.C1_TINY_F32, 64, 256, 704, 0),
]


@pytest.mark.parametrize("label,cfg,rows,d,ffn_,flags", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("residual", [False, True])
def test_chained_output_statistic(ffn, oracle_lib, label, cfg, rows, d, ffn_, flags, residual):
    import torch
    inp = synth.make_block_inputs(cfg, seed=60 + rows, rows=rows, d=d, ffn=ffn_)
    args = dev(inp, cfg.dtype)
    if flags & ffn.FFN_PREPARED_WEIGHTS:
        args[2:] = [ffn.ffn_prepare_weights(w) for w in args[2:]]
    if residual:
        flags |= ffn.FFN_RESIDUAL
    y, ss = ffn.ffn_block_forward_chained(*args, eps=cfg.eps, flags=flags)
    ref = ffn.ffn_block_forward(*args, eps=cfg.eps, flags=flags)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16) if y.dtype != torch.float32 else y,
                       ref.view(torch.int16) if ref.dtype != torch.float32 else ref)
    y_ref = oracle_lib.block_from_inputs(inp, residual=residual)
    y64 = to_host64(y)
    assert_dtype(y64, y_ref, cfg.dtype)
    check_sumsq(ss.cpu().numpy().astype(np.float64), y64, y_ref, 1e-4 if cfg.dtype == "f32" else BF16_MAX)
    ffn.ffn_device_status()


@pytest.mark.parametrize("label,cfg,rows,d,ffn_,flags", CASES, ids=[c[0] for c in CASES])
def test_chained_input_statistic(ffn, oracle_lib, label, cfg, rows, d, ffn_, flags):
    """The norm on a given sum of squares: the oracle's own statistic of x."""
    import torch
    import oracle
    inp = synth.make_block_inputs(cfg, seed=80 + rows, rows=rows, d=d, ffn=ffn_)
    args = dev(inp, cfg.dtype)
    if flags & ffn.FFN_PREPARED_WEIGHTS:
        args[2:] = [ffn.ffn_prepare_weights(w) for w in args[2:]]
    ss_x = oracle_lib.row_sumsq(oracle.widen(inp["x"], cfg.dtype)).astype(np.float32)
    y, _ = ffn.ffn_block_forward_chained(*args, eps=cfg.eps, flags=flags,
                                         x_sumsq=torch.from_numpy(ss_x).cuda(), y_sumsq=False)
    torch.cuda.synchronize()
    assert_dtype(to_host64(y), oracle_lib.block_from_inputs(inp), cfg.dtype)
    ffn.ffn_device_status()


@pytest.mark.parametrize("rows,d,ffn_", [(8, 1024, 2816), (640, 512, 1024)])
def test_two_block_chain(ffn, rows, d, ffn_):
    """Block 1 (skip connection) hands y and its row statistics to block 2;
    block 2 on the handed-on statistic against block 2 reducing the row
    itself: the same inputs, so the outputs agree within the bf16 bound of
    each other, and block 2's statistic describes its own y."""
    import torch
    cfg = synth.C3_DECODE_BF16
    inp1 = synth.make_block_inputs(cfg, seed=91, rows=rows, d=d, ffn=ffn_)
    inp2 = synth.make_block_inputs(cfg, seed=92, rows=rows, d=d, ffn=ffn_)
    a1, a2 = dev(inp1, "bf16"), dev(inp2, "bf16")
    R = ffn.FFN_RESIDUAL
    y1, ss1 = ffn.ffn_block_forward_chained(*a1, eps=cfg.eps, flags=R)
    y2, ss2 = ffn.ffn_block_forward_chained(y1, *a2[1:], eps=cfg.eps, flags=R, x_sumsq=ss1)
    y2_own = ffn.ffn_block_forward(y1, *a2[1:], eps=cfg.eps, flags=R)
    torch.cuda.synchronize()
    a, b = to_host64(y2), to_host64(y2_own)
    rms = float(np.sqrt(np.mean(b * b)))
    assert np.abs(a - b).max() <= 2e-2 * rms
    assert np.allclose(ss2.cpu().numpy(), np.sum(a * a, axis=1), rtol=1e-5, atol=0)
    ffn.ffn_device_status()


def test_chained_rejects_overlapping_statistic(ffn):
    import torch
    from transformer_ffn_rmsnorm_gb300 import _lib
    inp = synth.make_block_inputs(synth.C3_DECODE_BF16, seed=1, rows=4, d=256, ffn=512)
    x, g, wg, wu, wd = dev(inp, "bf16")
    y = torch.empty_like(x)
    ws = ffn.workspace(ffn.ffn_block_workspace_bytes(4, 256, 512, torch.bfloat16), x.device)
    st = _lib.load().ffn_block_forward_chained(*[ffn._ptr(t) for t in (x, None, g, wg, wu, wd, y)],
                                               ffn._ptr(y), 4, 256, 512, 1e-5, _lib.FFN_BF16, 0,
                                               ffn._ptr(ws), ws.numel(), None)
    assert st == _lib.FFN_ERR_ALIAS
