"""The C ABI on the host (CPU only): the library loads, exports every symbol
include/ffn.h declares, and rejects bad arguments before touching CUDA."""

import ctypes
import os
import re

import numpy as np
import pytest

import synth
from transformer_ffn_rmsnorm_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ffn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(ffn_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for n in ("ffn_rmsnorm", "ffn_swiglu", "ffn_block_forward", "ffn_block_forward_q4"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks a signature for {name}"


def test_status_strings(lib):
    for code in range(11):
        s = lib.ffn_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.ffn_status_string(99).decode() == "unknown status"


def test_null_and_shape_errors_without_gpu(lib):
    p = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    assert lib.ffn_rmsnorm(None, p, p, 1, 8, 1e-5, _lib.FFN_BF16, None) == _lib.FFN_ERR_NULL
    assert lib.ffn_rmsnorm(p, p, ctypes.c_void_p(8192), -1, 8, 1e-5, _lib.FFN_BF16, None) == _lib.FFN_ERR_SHAPE
    assert lib.ffn_rmsnorm(p, p, ctypes.c_void_p(8192), 1, 0, 1e-5, _lib.FFN_BF16, None) == _lib.FFN_ERR_SHAPE
    assert lib.ffn_rmsnorm(p, p, ctypes.c_void_p(8192), 1, 8, 1e-5, 7, None) == _lib.FFN_ERR_DTYPE
    assert lib.ffn_rmsnorm(ctypes.c_void_p(4098), p, ctypes.c_void_p(8192), 1, 8, 1e-5, _lib.FFN_BF16,
                           None) == _lib.FFN_ERR_ALIGN
    assert lib.ffn_swiglu(p, None, p, 4, _lib.FFN_F16, None) == _lib.FFN_ERR_NULL
    assert lib.ffn_swiglu(p, p, p, -4, _lib.FFN_F16, None) == _lib.FFN_ERR_SHAPE
    # h overlapping gate at an offset (not in place) is rejected
    assert lib.ffn_swiglu(ctypes.c_void_p(4096), ctypes.c_void_p(1 << 20), ctypes.c_void_p(4096 + 16),
                          64, _lib.FFN_F16, None) == _lib.FFN_ERR_ALIAS
    # empty inputs are valid and launch nothing
    assert lib.ffn_rmsnorm(p, ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 21), 0, 8, 1e-5,
                           _lib.FFN_BF16, None) == _lib.FFN_OK
    assert lib.ffn_swiglu(p, ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 21), 0, _lib.FFN_F16,
                          None) == _lib.FFN_OK


def _ws(lib, rows, d, ffn, dt, flags=0):
    out = ctypes.c_size_t(0)
    st = lib.ffn_block_workspace_bytes(rows, d, ffn, dt, flags, ctypes.byref(out))
    return st, out.value


def test_workspace_query(lib):
    st, n = _ws(lib, 8, 4096, 14336, _lib.FFN_BF16)
    assert st == 0 and n > 0
    st, n2 = _ws(lib, 4096, 4096, 11008, _lib.FFN_BF16)
    assert st == 0 and n2 >= 4096 * (4096 + 11008) * 2
    st, n3 = _ws(lib, 4096, 4096, 11008, _lib.FFN_BF16, _lib.FFN_GATEUP_UNFUSED)
    assert st == 0 and n3 >= n2 + 2 * 4096 * 11008 * 2
    assert _ws(lib, 0, 4096, 11008, _lib.FFN_BF16) == (0, 0)
    assert _ws(lib, 4, 4100, 11008, _lib.FFN_BF16)[0] == _lib.FFN_ERR_SHAPE       # d % 8
    assert _ws(lib, 4, 4096, 11008, _lib.FFN_F32, _lib.FFN_PATH_GEMM)[0] == _lib.FFN_ERR_FLAGS
    assert _ws(lib, 4, 4096, 11008, _lib.FFN_BF16, 3)[0] == _lib.FFN_ERR_FLAGS      # fused+unfused
    assert _ws(lib, 4, 4096, 11008, _lib.FFN_BF16, 1 << 20)[0] == _lib.FFN_ERR_FLAGS
    assert _ws(lib, 65, 4096, 11008, _lib.FFN_BF16, _lib.FFN_PATH_GEMV)[0] == _lib.FFN_ERR_SHAPE
    assert _ws(lib, 64, 4096, 11008, _lib.FFN_BF16, _lib.FFN_PATH_GEMV)[0] == 0
    out = ctypes.c_size_t(0)
    assert lib.ffn_block_q4_workspace_bytes(8, 5120, 17408, ctypes.byref(out)) == 0 and out.value > 0
    assert lib.ffn_block_q4_workspace_bytes(8, 5000, 17408, ctypes.byref(out)) == _lib.FFN_ERR_SHAPE   # in % 32
    assert lib.ffn_block_q4_workspace_bytes(8, 5024, 17408, ctypes.byref(out)) == 0            # whole blocks
    assert lib.ffn_block_q4_workspace_bytes(8, 5120, 17400, ctypes.byref(out)) == _lib.FFN_ERR_SHAPE


def test_block_forward_rejects_before_launch(lib):
    p = [ctypes.c_void_p((i + 1) << 24) for i in range(8)]
    # workspace too small
    assert lib.ffn_block_forward(*p[:6], 8, 4096, 14336, 1e-5, _lib.FFN_BF16, 0, p[6], 16,
                                 None) == _lib.FFN_ERR_WORKSPACE
    # y aliases x
    st, need = _ws(lib, 8, 64, 128, _lib.FFN_BF16)
    assert lib.ffn_block_forward(p[0], p[1], p[2], p[3], p[4], p[0], 8, 64, 128, 1e-5, _lib.FFN_BF16,
                                 0, p[6], need, None) == _lib.FFN_ERR_ALIAS
    # misaligned weight
    assert lib.ffn_block_forward(p[0], p[1], ctypes.c_void_p((3 << 24) + 8), p[3], p[4], p[5], 8, 64,
                                 128, 1e-5, _lib.FFN_BF16, 0, p[6], need, None) == _lib.FFN_ERR_ALIGN
    q = _lib.Q4Weight(p[2].value, p[3].value)
    assert lib.ffn_block_forward_q4(p[0], p[1], q, q, q, p[5], 8, 512, 1024, 1e-6, 1, p[6], 1 << 30,
                                    None) == _lib.FFN_ERR_FLAGS


@pytest.mark.parametrize("d,ffn_", [(256, 384), (96, 160), (416, 224)])
def test_q4_pack_host_matches_layout(lib, d, ffn_):
    """The library's packer writes the bytes of the documented layout, the
    padding of a last, partial group included (zero bytes, zero scales)."""
    from transformer_ffn_rmsnorm_gb300 import ffn
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=4, rows=1, d=d, ffn=ffn_)
    for name in ("gate", "down"):
        qs, sc = ffn.ffn_q4_pack_host(inp["q_" + name], inp["s_" + name].view(np.uint16))
        assert np.array_equal(qs, inp["qs_" + name])
        assert np.array_equal(sc, inp["sc_" + name])
    bad = inp["q_gate"].copy()
    bad[0, 0] = 8
    with pytest.raises(Exception):
        ffn.ffn_q4_pack_host(bad, inp["s_gate"].view(np.uint16))


def test_launch_counter_starts_quiet(lib):
    before = lib.ffn_launch_count()
    p = ctypes.c_void_p(4096)
    lib.ffn_rmsnorm(None, p, p, 1, 8, 1e-5, _lib.FFN_BF16, None)
    assert lib.ffn_launch_count() == before   # rejected calls launch nothing


def test_kernel_names(lib):
    n = lib.ffn_kernel_kinds()
    names = [lib.ffn_kernel_name(k).decode() for k in range(n)]
    assert "gemm_gateup" in names and "rmsnorm" in names and len(set(names)) == n


def test_prepare_weights_rejects_before_launch(lib):
    p = ctypes.c_void_p(4096)
    assert lib.ffn_prepare_weights(None, p, 8, _lib.FFN_BF16, None) == _lib.FFN_ERR_NULL
    assert lib.ffn_prepare_weights(p, ctypes.c_void_p(1 << 20), 8, _lib.FFN_F32, None) == _lib.FFN_ERR_DTYPE
    assert lib.ffn_prepare_weights(p, ctypes.c_void_p(1 << 20), -1, _lib.FFN_BF16, None) == _lib.FFN_ERR_SHAPE
    assert lib.ffn_prepare_weights(p, ctypes.c_void_p(4096 + 16), 64, _lib.FFN_BF16, None) == _lib.FFN_ERR_ALIAS
    assert lib.ffn_prepare_weights(None, None, 0, _lib.FFN_BF16, None) == _lib.FFN_OK
    out = ctypes.c_size_t(0)
    flags = _lib.FFN_PREPARED_WEIGHTS
    assert lib.ffn_block_workspace_bytes(4096, 4096, 11008, _lib.FFN_BF16, flags, ctypes.byref(out)) == 0
    assert out.value >= 4096 * (4096 + 11008) * 2
    assert lib.ffn_block_workspace_bytes(8, 64, 64, _lib.FFN_F32, flags, ctypes.byref(out)) == _lib.FFN_ERR_FLAGS
    assert lib.ffn_block_workspace_bytes(8, 64, 64, _lib.FFN_BF16, flags | _lib.FFN_ACT_SPLIT,
                                         ctypes.byref(out)) == _lib.FFN_ERR_FLAGS


def test_host_block_entry_rejects_before_launch(lib):
    out = ctypes.c_size_t(0)
    assert lib.ffn_block_host_workspace_bytes(0, 4096, 11008, _lib.FFN_BF16, 0, ctypes.byref(out)) == 0
    assert out.value == 0
    assert lib.ffn_block_host_workspace_bytes(4096, 4096, 11008, _lib.FFN_BF16, 0, ctypes.byref(out)) == 0
    staged = 2 * 4096 * 4096 * 2
    blk = ctypes.c_size_t(0)
    assert lib.ffn_block_workspace_bytes(1024, 4096, 11008, _lib.FFN_BF16, 0, ctypes.byref(blk)) == 0
    assert out.value >= staged + blk.value
    assert lib.ffn_block_host_workspace_bytes(8, 4100, 11008, _lib.FFN_BF16, 0,
                                              ctypes.byref(out)) == _lib.FFN_ERR_SHAPE
    p = [ctypes.c_void_p((i + 1) << 24) for i in range(8)]
    need = ctypes.c_size_t(0)
    lib.ffn_block_host_workspace_bytes(8, 64, 128, _lib.FFN_BF16, 0, ctypes.byref(need))
    # NULL host buffer, workspace too small, overlapping host buffers
    assert lib.ffn_block_forward_host(None, *p[1:5], p[5], 8, 64, 128, 1e-5, _lib.FFN_BF16, 0, p[6],
                                      need.value, None) == _lib.FFN_ERR_NULL
    assert lib.ffn_block_forward_host(*p[:6], 8, 64, 128, 1e-5, _lib.FFN_BF16, 0, p[6], 16,
                                      None) == _lib.FFN_ERR_WORKSPACE
    x = ctypes.c_void_p(1 << 30)
    assert lib.ffn_block_forward_host(x, *p[1:5], ctypes.c_void_p((1 << 30) + 512), 8, 64, 128, 1e-5,
                                      _lib.FFN_BF16, 0, p[6], need.value, None) == _lib.FFN_ERR_ALIAS


def test_residual_flag_accepted_by_the_planner(lib):
    out = ctypes.c_size_t(0)
    assert lib.ffn_block_workspace_bytes(4096, 4096, 11008, _lib.FFN_BF16, _lib.FFN_RESIDUAL,
                                         ctypes.byref(out)) == 0
    assert lib.ffn_block_workspace_bytes(8, 4096, 11008, _lib.FFN_BF16,
                                         _lib.FFN_RESIDUAL | _lib.FFN_PREPARED_WEIGHTS, ctypes.byref(out)) == 0
    assert lib.ffn_block_workspace_bytes(8, 64, 64, _lib.FFN_F32, _lib.FFN_RESIDUAL, ctypes.byref(out)) == 0


def test_fp8_entry_rejects_before_launch(lib):
    out = ctypes.c_size_t(0)
    assert lib.ffn_block_fp8_workspace_bytes(8, 4096, 14336, ctypes.byref(out)) == 0 and out.value > 0
    assert lib.ffn_block_fp8_workspace_bytes(0, 4096, 14336, ctypes.byref(out)) == 0 and out.value == 0
    for d, f in ((4160, 14336), (4096, 14400), (4096 + 128, 14336), (128, 256), (256, 128)):   # multiples of 256
        assert lib.ffn_block_fp8_workspace_bytes(8, d, f, ctypes.byref(out)) == _lib.FFN_ERR_SHAPE
    assert lib.ffn_block_fp8_workspace_bytes(-1, 256, 256, ctypes.byref(out)) == _lib.FFN_ERR_SHAPE
    p = [ctypes.c_void_p((i + 1) << 24) for i in range(12)]
    w = [_lib.Fp8Weight(p[2 + 2 * i].value, p[3 + 2 * i].value) for i in range(3)]
    lib.ffn_block_fp8_workspace_bytes(8, 512, 1024, ctypes.byref(out))
    need = out.value
    # missing scale pointer, unknown flag, short workspace, misaligned codes, y aliasing the codes
    bad = _lib.Fp8Weight(p[2].value, None)
    assert lib.ffn_block_forward_fp8(p[0], p[1], bad, w[1], w[2], p[8], 8, 512, 1024, 1e-6, 0, p[9], need,
                                     None) == _lib.FFN_ERR_NULL
    assert lib.ffn_block_forward_fp8(p[0], p[1], *w, p[8], 8, 512, 1024, 1e-6, _lib.FFN_PATH_GEMM, p[9],
                                     need, None) == _lib.FFN_ERR_FLAGS
    assert lib.ffn_block_forward_fp8(p[0], p[1], *w, p[8], 8, 512, 1024, 1e-6, 0, p[9], need - 1,
                                     None) == _lib.FFN_ERR_WORKSPACE
    mis = _lib.Fp8Weight(p[2].value + 8, p[3].value)
    assert lib.ffn_block_forward_fp8(p[0], p[1], mis, w[1], w[2], p[8], 8, 512, 1024, 1e-6, 0, p[9], need,
                                     None) == _lib.FFN_ERR_ALIGN
    assert lib.ffn_block_forward_fp8(p[0], p[1], *w, ctypes.c_void_p(p[4].value + 4096), 8, 512, 1024, 1e-6,
                                     0, p[9], need, None) == _lib.FFN_ERR_ALIAS


def test_quantised_prepare_rejects_before_launch(lib):
    p = [ctypes.c_void_p((i + 1) << 24) for i in range(6)]
    f = _lib.Fp8Weight(p[0].value, p[1].value)
    q = _lib.Q4Weight(p[0].value, p[1].value)
    assert lib.ffn_prepare_weights_fp8(f, p[2], 4, 24, None) == _lib.FFN_ERR_SHAPE       # in % 16
    assert lib.ffn_prepare_weights_q4(q, p[2], 4, 48, None) == _lib.FFN_ERR_SHAPE        # in % 32
    assert lib.ffn_prepare_weights_fp8(_lib.Fp8Weight(p[0].value, None), p[2], 4, 32, None) == _lib.FFN_ERR_NULL
    assert lib.ffn_prepare_weights_fp8(f, ctypes.c_void_p(p[2].value + 8), 4, 32, None) == _lib.FFN_ERR_ALIGN
    assert lib.ffn_prepare_weights_fp8(f, ctypes.c_void_p(p[0].value + 64), 4, 32, None) == _lib.FFN_ERR_ALIAS
    assert lib.ffn_prepare_weights_q4(q, ctypes.c_void_p(p[1].value), 4, 128, None) == _lib.FFN_ERR_ALIAS
    assert lib.ffn_prepare_weights_fp8(f, p[2], 0, 32, None) == _lib.FFN_OK


def test_q8_entry_rejects_before_launch(lib):
    out = ctypes.c_size_t(0)
    assert lib.ffn_block_q8_workspace_bytes(8, 4096, 14336, ctypes.byref(out)) == 0 and out.value > 0
    for d, f in ((4096 + 128, 14336), (4096, 14336 + 128)):   # multiples of 256 only
        assert lib.ffn_block_q8_workspace_bytes(8, d, f, ctypes.byref(out)) == _lib.FFN_ERR_SHAPE
    p = [ctypes.c_void_p((i + 1) << 24) for i in range(12)]
    w = [_lib.Q8Weight(p[2 + 2 * i].value, p[3 + 2 * i].value) for i in range(3)]
    lib.ffn_block_q8_workspace_bytes(8, 512, 1024, ctypes.byref(out))
    need = out.value
    assert lib.ffn_block_forward_q8(p[0], p[1], _lib.Q8Weight(p[2].value, None), w[1], w[2], p[8], 8, 512, 1024,
                                    1e-6, 0, p[9], need, None) == _lib.FFN_ERR_NULL
    assert lib.ffn_block_forward_q8(p[0], p[1], *w, p[8], 8, 512, 1024, 1e-6, _lib.FFN_GATEUP_FUSED, p[9], need,
                                    None) == _lib.FFN_ERR_FLAGS
    assert lib.ffn_block_forward_q8(p[0], p[1], *w, p[8], 8, 512, 1024, 1e-6, 0, p[9], need - 1,
                                    None) == _lib.FFN_ERR_WORKSPACE
    assert lib.ffn_block_forward_q8(p[0], p[1], *w, ctypes.c_void_p(p[3].value + 256), 8, 512, 1024, 1e-6, 0, p[9],
                                    need, None) == _lib.FFN_ERR_ALIAS
    q = _lib.Q8Weight(p[0].value, p[1].value)
    assert lib.ffn_prepare_weights_q8(q, p[2], 4, 48, None) == _lib.FFN_ERR_SHAPE        # in % 32
    assert lib.ffn_prepare_weights_q8(q, ctypes.c_void_p(p[1].value + 32), 64, 64, None) == _lib.FFN_ERR_ALIAS
