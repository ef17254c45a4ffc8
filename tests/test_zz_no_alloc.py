"""ffn_block_forward_decode_static: the decode block for callers that cannot
pass a workspace (its scratch is a fixed device array inside the library).

Checked through the C ABI, call after call, against ffn_block_forward (which
takes a caller's workspace) bit for bit -- both run the same kernels in the
same operand mode on the same inputs -- and against the float64 oracle
within the bf16 bound.  The calls go from the largest shape to the smallest
and from bf16 (two-term fragments) to fp16, so every later call reads
scratch regions an earlier, larger call has filled: stale bytes would show
up as a bitwise difference.  One call runs at the documented limit.  This
file is collected last on purpose."""

import ctypes

import numpy as np
import pytest

import synth
from gpu_util import assert_lowp, to_dev, to_host64

pytestmark = pytest.mark.gpu


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _call_static(lib, args, y, rows, d, ffn, eps, dt):
    p = [ctypes.c_void_p(t.data_ptr()) for t in args]
    return lib.ffn_block_forward_decode_static(*p, ctypes.c_void_p(y.data_ptr()), rows, d, ffn, eps, dt, _stream())


def _f16_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run_case(lib, ffn, oracle_lib, cfg, seed):
    import torch
    from transformer_ffn_rmsnorm_gb300 import _lib
    inp = synth.make_block_inputs(cfg, seed=seed)
    names = ("x", "g", "w_gate", "w_up", "w_down")
    if cfg.dtype == "bf16":
        args, code = [to_dev(inp[k], "bf16") for k in names], _lib.FFN_BF16
    else:
        args, code = [_f16_dev(inp[k]) for k in names], _lib.FFN_F16
    y = torch.full_like(args[0], float("nan"))
    st = _call_static(lib, args, y, cfg.rows, cfg.d, cfg.ffn, cfg.eps, code)
    assert st == _lib.FFN_OK, _lib.STATUS[st]
    ref = ffn.ffn_block_forward(*args, eps=cfg.eps)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), "static scratch result differs from the workspace entry point"
    assert_lowp(to_host64(y), oracle_lib.block_from_inputs(inp))


def test_static_scratch_matches_workspace_entry_point_and_oracle(oracle_lib):
    from transformer_ffn_rmsnorm_gb300 import _lib, ffn
    lib = _lib.load()
    cases = [synth.BlockConfig("a", 16, 1024, 2816, 1e-5, "bf16"),   # two token tiles, two-term fragments
             synth.BlockConfig("b", 5, 520, 4104, 1e-5, "bf16"),     # ragged d and ffn, one tile
             synth.BlockConfig("c", 11, 768, 2048, 1e-5, "f16")]     # one-term fragments
    for i, cfg in enumerate(cases):   # calls in a row, each smaller than the one before
        _run_case(lib, ffn, oracle_lib, cfg, seed=40 + i)
    ffn.ffn_device_status()


def test_static_scratch_at_its_limit(oracle_lib):
    """rows 16, d 8192, ffn 32768 in bf16 (two-term fragments): the largest
    shape the entry point documents fits its fixed array."""
    from transformer_ffn_rmsnorm_gb300 import _lib, ffn
    lib = _lib.load()
    _run_case(lib, ffn, oracle_lib, synth.BlockConfig("limit", 16, 8192, 32768, 1e-5, "bf16"), seed=44)
    ffn.ffn_device_status()


def test_static_scratch_rejects_sizes_beyond_its_limits():
    import torch
    from transformer_ffn_rmsnorm_gb300 import _lib
    lib = _lib.load()
    buf = torch.zeros(1 << 16, dtype=torch.bfloat16, device="cuda")
    p = [ctypes.c_void_p(buf.data_ptr() + 4096 * i) for i in range(6)]
    for rows, d, ffn_ in ((17, 64, 64), (1, 8200, 64), (1, 64, 32776)):
        st = lib.ffn_block_forward_decode_static(*p, rows, d, ffn_, 1e-5, _lib.FFN_BF16, None)
        assert st == _lib.FFN_ERR_SHAPE
    assert lib.ffn_block_forward_decode_static(*p, 1, 64, 64, 1e-5, _lib.FFN_F32, None) == _lib.FFN_ERR_DTYPE
