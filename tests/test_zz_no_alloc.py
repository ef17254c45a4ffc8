"""ffn_block_forward_decode_static: the decode block for callers that cannot
pass a workspace (its scratch is a fixed device array inside the library).

Checked through the C ABI against ffn_block_forward (which takes a caller's
workspace) on two calls in a row with different shapes, so the second call
also shows that what the first left in the shared array does not leak into
its result.  This file is collected last on purpose."""

import ctypes

import numpy as np
import pytest

import synth
from gpu_util import assert_lowp, to_dev, to_host64

pytestmark = pytest.mark.gpu


def _call_static(lib, args, y, rows, d, ffn, eps, dt):
    import torch
    p = [ctypes.c_void_p(t.data_ptr()) for t in args]
    st = lib.ffn_block_forward_decode_static(*p, ctypes.c_void_p(y.data_ptr()), rows, d, ffn, eps, dt,
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def test_static_scratch_matches_workspace_entry_point():
    import torch
    from transformer_ffn_rmsnorm_gb300 import _lib, ffn
    lib = _lib.load()
    cases = [synth.BlockConfig("a", 8, 1024, 2816, 1e-5, "bf16"),
             synth.BlockConfig("b", 13, 520, 4104, 1e-5, "bf16")]
    for i, cfg in enumerate(cases):   # two calls in a row, different shapes
        inp = synth.make_block_inputs(cfg, seed=40 + i)
        args = [to_dev(inp[k], "bf16") for k in ("x", "g", "w_gate", "w_up", "w_down")]
        ref = ffn.ffn_block_forward(*args, eps=cfg.eps)
        y = torch.full_like(ref, float("nan"))
        st = _call_static(lib, args, y, cfg.rows, cfg.d, cfg.ffn, cfg.eps, _lib.FFN_BF16)
        assert st == _lib.FFN_OK, _lib.STATUS[st]
        torch.cuda.synchronize()
        assert_lowp(to_host64(y), to_host64(ref))
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
