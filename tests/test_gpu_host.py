"""ffn_block_forward_host: x and y in host memory, copies overlapped with the
compute in row chunks.  Checked against the float64 oracle and, where every
chunk takes the same path as the whole batch, byte for byte against
ffn_block_forward on device buffers (rows are independent: chunking changes
no output's arithmetic)."""

import numpy as np
import pytest

import synth
from gpu_util import assert_lowp, to_dev, to_host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ffn():
    from transformer_ffn_rmsnorm_gb300 import ffn as m
    return m


def host_bf16(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()


@pytest.mark.parametrize("rows", [8, 300, 3500, 9000])
@pytest.mark.parametrize("prepared", [False, True])
def test_host_block_matches_device_block(ffn, oracle_lib, rows, prepared):
    """3500 rows: chunks of 2476 and 1024 rows; 9000 rows: 4096, 3880 and
    1024; all through the tensor-core path (every tile sums its whole K in
    the same order, so the chunked result is bitwise the one-call result)."""
    import torch
    inp = synth.make_block_inputs(synth.C4_PREFILL_BF16, seed=rows, rows=rows, d=256, ffn=384)
    g = to_dev(inp["g"], "bf16")
    w = [to_dev(inp[k], "bf16") for k in ("w_gate", "w_up", "w_down")]
    flags = 0
    if prepared:
        w = [ffn.ffn_prepare_weights(t) for t in w]
        flags = ffn.FFN_PREPARED_WEIGHTS
    xh = host_bf16(inp["x"])   # alive until the stream has passed the call
    y_host = ffn.ffn_block_forward_host(xh, g, *w, eps=inp["cfg"].eps, flags=flags)
    torch.cuda.current_stream().synchronize()
    y_dev = ffn.ffn_block_forward(to_dev(inp["x"], "bf16"), g, *w, eps=inp["cfg"].eps, flags=flags)
    assert torch.equal(y_host.view(torch.int16), y_dev.cpu().view(torch.int16))
    assert_lowp(to_host64(y_host), oracle_lib.block_from_inputs(inp))
    ffn.ffn_device_status()


@pytest.mark.parametrize("total", [1034, 2058])
def test_host_block_short_chunk(ffn, oracle_lib, total):
    """1034 rows: chunks of 10 and 1024, the first on the decode path; 2058
    rows: 1034 and 1024."""
    import torch
    inp = synth.make_block_inputs(synth.C4_PREFILL_BF16, seed=9, rows=total, d=512, ffn=704)
    args = [to_dev(inp[k], "bf16") for k in ("g", "w_gate", "w_up", "w_down")]
    xh = host_bf16(inp["x"])   # alive until the stream has passed the call
    y = ffn.ffn_block_forward_host(xh, *args, eps=inp["cfg"].eps)
    torch.cuda.current_stream().synchronize()
    got = to_host64(y)
    rows = np.unique(np.r_[0:40, 1015:1040, total - 30:total])
    rows = rows[rows < total]
    ref = oracle_lib.block_from_inputs(inp, rows=rows)
    assert_lowp(got[rows], ref)
    ffn.ffn_device_status()


def test_host_block_calls_in_a_row_and_empty(ffn):
    """Back-to-back calls on one workspace use its two staging sets in turn:
    the third call's input copies must wait until the first call has
    computed from that set, and its compute until the first call's output
    copies have drained it.  An empty batch is valid and queues nothing."""
    import torch
    inps = [synth.make_block_inputs(synth.C4_PREFILL_BF16, seed=3 + k, rows=2600, d=256, ffn=384)
            for k in range(4)]
    args = [to_dev(inps[0][k], "bf16") for k in ("g", "w_gate", "w_up", "w_down")]
    ws = ffn.workspace(ffn.ffn_block_host_workspace_bytes(2600, 256, 384, torch.bfloat16), torch.device("cuda"))
    xs = [host_bf16(inp["x"]) for inp in inps]   # kept alive until the copies have run
    ys = [ffn.ffn_block_forward_host(x, *args, eps=1e-6, ws=ws) for x in xs]
    torch.cuda.current_stream().synchronize()
    for inp, y in zip(inps, ys):
        r = ffn.ffn_block_forward(to_dev(inp["x"], "bf16"), *args, eps=1e-6).cpu()
        assert torch.equal(y.view(torch.int16), r.view(torch.int16))
    e = torch.empty((0, 256), dtype=torch.bfloat16).pin_memory()
    assert ffn.ffn_block_forward_host(e, *args, eps=1e-6).numel() == 0
    ffn.ffn_device_status()


def test_host_block_at_the_benchmark_shape(ffn, oracle_lib):
    """The timed end-to-end call itself: 4096 tokens, d 4096 -> ffn 11008,
    prepared weights, chunks of 3072 and 1024 rows, three calls in a row on
    one workspace (both staging sets, the first one twice).  Bitwise against
    one ffn_block_forward of the whole batch on device buffers; sampled rows
    (both ends of each chunk and its middle) against the float64 oracle."""
    import torch
    inp = synth.make_block_inputs(synth.C4_PREFILL_BF16, seed=0)
    cfg = inp["cfg"]
    assert (cfg.rows, cfg.d, cfg.ffn) == (4096, 4096, 11008)
    g = to_dev(inp["g"], "bf16")
    w = [ffn.ffn_prepare_weights(to_dev(inp[k], "bf16")) for k in ("w_gate", "w_up", "w_down")]
    flags = ffn.FFN_PREPARED_WEIGHTS
    ws = ffn.workspace(ffn.ffn_block_host_workspace_bytes(cfg.rows, cfg.d, cfg.ffn, torch.bfloat16, flags),
                       torch.device("cuda"))
    xh = host_bf16(inp["x"])   # alive until the stream has passed the calls
    ys = [ffn.ffn_block_forward_host(xh, g, *w, eps=cfg.eps, flags=flags, ws=ws) for _ in range(3)]
    torch.cuda.current_stream().synchronize()
    y_dev = ffn.ffn_block_forward(to_dev(inp["x"], "bf16"), g, *w, eps=cfg.eps, flags=flags).cpu()
    for y in ys:
        assert torch.equal(y.view(torch.int16), y_dev.view(torch.int16))
    rows = np.r_[0:4, 1534:1538, 3068:3076, 3582:3586, 4092:4096]
    assert_lowp(to_host64(ys[-1])[rows], oracle_lib.block_from_inputs(inp, rows=rows))
    ffn.ffn_device_status()
