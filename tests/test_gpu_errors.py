"""Argument errors with real device buffers: rejected on the host, nothing
launched, and the device stays usable."""

import ctypes

import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    from transformer_ffn_rmsnorm_gb300 import _lib, ffn
    return torch, _lib, ffn


def test_misaligned_and_aliased(env):
    torch, _lib, ffn = env
    L = _lib.load()
    buf = torch.zeros(1 << 20, dtype=torch.bfloat16, device="cuda")
    p = buf.data_ptr()
    before = ffn.ffn_launch_count()
    st = L.ffn_rmsnorm(ctypes.c_void_p(p + 2), ctypes.c_void_p(p + 4096), ctypes.c_void_p(p + 8192),
                       2, 64, 1e-5, _lib.FFN_BF16, None)
    assert st == _lib.FFN_ERR_ALIGN
    st = L.ffn_rmsnorm(ctypes.c_void_p(p), ctypes.c_void_p(p + 65536), ctypes.c_void_p(p + 64),
                       2, 64, 1e-5, _lib.FFN_BF16, None)
    assert st == _lib.FFN_ERR_ALIAS
    with pytest.raises(ffn.FFNError):
        x = buf[: 8 * 64].view(8, 64)
        w = buf[4096: 4096 + 128 * 64].view(128, 64)
        wd = buf[16384: 16384 + 128 * 64].view(64, 128)
        ffn.ffn_block_forward(x, buf[100000:100064], w, w, wd, eps=1e-5, out=x)
    assert ffn.ffn_launch_count() == before
    torch.cuda.synchronize()
    ffn.ffn_device_status()


def test_unsupported_dtype_tensor(env):
    torch, _lib, ffn = env
    x = torch.zeros((2, 8), dtype=torch.float64, device="cuda")
    with pytest.raises(TypeError):
        ffn.ffn_rmsnorm(x, x[0], eps=1e-5)


def test_bounded_wait_gives_up_and_device_stays_usable(env):
    """A wait that nothing completes ends after its limit with FFN_ERR_TIMEOUT
    in the status word; a second role with a 1000x longer limit is released by
    the abort flag; the next call on the same context computes correctly."""
    import time
    import numpy as np
    torch, _lib, ffn = env
    torch.cuda.synchronize()
    ffn.ffn_device_status()                      # start from a clean status word
    limit_ns = 2_000_000                         # 2 ms (the second role: 2 s)
    t0 = time.perf_counter()
    ffn.ffn_selftest_bounded_wait(limit_ns)
    with pytest.raises(ffn.FFNError) as err:
        ffn.ffn_device_status()
    elapsed = time.perf_counter() - t0
    assert err.value.status == _lib.FFN_ERR_TIMEOUT
    assert elapsed < 0.5, elapsed               # far below the second role's 2 s
    ffn.ffn_device_status()                      # the word was cleared by the read
    x = torch.randn(4, 256, device="cuda")
    g = torch.ones(256, device="cuda")
    n = ffn.ffn_rmsnorm(x, g, eps=1e-6)
    ref = x / torch.sqrt((x * x).mean(dim=1, keepdim=True) + 1e-6)
    assert np.allclose(n.cpu().numpy(), ref.cpu().numpy(), rtol=1e-5, atol=1e-6)
    ffn.ffn_device_status()
