"""ffn_rmsnorm and ffn_swiglu on the GPU against the float64 oracle."""

import numpy as np
import pytest

import synth
from gpu_util import assert_lowp, errors, to_dev, to_host64
from oracle import widen

pytestmark = pytest.mark.gpu

# Per-element bound for one rounding of an fp32 result to the storage type:
# half an ulp is at most 2^-8 |v| (bf16), 2^-11 |v| (fp16) of the value, plus
# the fp32 arithmetic before it (relative) and the subnormal spacing (absolute).
ROUNDING = {"bf16": (2.0 ** -8, 1e-5, 1e-38), "f16": (2.0 ** -11, 1e-5, 2.0 ** -25),
            "f32": (0.0, 2e-5, 1e-30)}


def assert_rounded(got, ref, dtype):
    half_ulp, arith, tiny = ROUNDING[dtype]
    assert np.all(np.isfinite(got))
    bound = (half_ulp + arith) * np.abs(ref) + tiny
    bad = np.abs(got - ref) > bound
    assert not bad.any(), (f"{int(bad.sum())} elements beyond one {dtype} rounding, e.g. got "
                           f"{got[bad][:3]} for {ref[bad][:3]}")


@pytest.fixture(scope="module")
def ffn():
    from transformer_ffn_rmsnorm_gb300 import ffn as m
    return m


NORM_SHAPES = [(1, 8), (3, 40), (5, 36), (17, 256), (33, 4096), (4, 12288), (2, 16384),
               (2, 33000), (1, 40000)]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("rows,d", NORM_SHAPES)
def test_rmsnorm(ffn, oracle_lib, dtype, rows, d):
    if dtype == "f32" and d % 4:
        d += 4 - d % 4
    cfg = synth.NormConfig("t", rows, d, 1e-5, dtype)
    inp = synth.make_norm_inputs(cfg, seed=rows * 7 + d)
    n = ffn.ffn_rmsnorm(to_dev(inp["x"], dtype), to_dev(inp["g"], dtype), eps=1e-5)
    ref = oracle_lib.rmsnorm(widen(inp["x"], dtype), widen(inp["g"], dtype), 1e-5)
    assert_rounded(to_host64(n), ref, dtype)


def test_rmsnorm_in_place_and_empty(ffn, oracle_lib):
    import torch
    inp = synth.make_norm_inputs(synth.C2A_RMSNORM_F16, seed=1, rows=9, d=4096)
    x = to_dev(inp["x"], "f16")
    ffn.ffn_rmsnorm(x, to_dev(inp["g"], "f16"), eps=1e-5, out=x)
    ref = oracle_lib.rmsnorm(widen(inp["x"], "f16"), widen(inp["g"], "f16"), 1e-5)
    assert_lowp(to_host64(x), ref)
    e = torch.empty((0, 64), dtype=torch.float16, device="cuda")
    assert ffn.ffn_rmsnorm(e, torch.ones(64, dtype=torch.float16, device="cuda"), eps=1e-5).numel() == 0


def test_rmsnorm_constant_and_zero_rows(ffn):
    import torch
    x = torch.zeros((3, 512), dtype=torch.bfloat16, device="cuda")
    x[1] = 2.5
    x[2] = -0.75
    g = torch.full((512,), 1.5, dtype=torch.bfloat16, device="cuda")
    n = ffn.ffn_rmsnorm(x, g, eps=1e-6).float().cpu().numpy()
    assert np.all(n[0] == 0.0)
    assert np.allclose(n[1], 1.5, rtol=2 ** -8) and np.allclose(n[2], -1.5, rtol=2 ** -8)


def test_rmsnorm_full_size_fp16(ffn, oracle_lib):
    """16384 x 4096 fp16, eps 1e-5: sampled rows checked against the oracle."""
    inp = synth.make_norm_inputs(synth.C2A_RMSNORM_F16, seed=0)
    n = ffn.ffn_rmsnorm(to_dev(inp["x"], "f16"), to_dev(inp["g"], "f16"), eps=1e-5)
    rows = np.unique(np.concatenate([[0, 1, 8191, 16383], np.random.default_rng(0).integers(0, 16384, 60)]))
    ref = oracle_lib.rmsnorm(widen(inp["x"][rows], "f16"), widen(inp["g"], "f16"), 1e-5)
    got = to_host64(n[rows])
    assert_lowp(got, ref)              # the bf16 bound, applied to the fp16 workload
    assert_rounded(got, ref, "f16")    # and one fp16 rounding per element


SWIGLU_COUNTS = [1, 7, 8, 9, 4096, 1000003]


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("count", SWIGLU_COUNTS)
def test_swiglu(ffn, oracle_lib, dtype, count):
    cfg = synth.SwigluConfig("t", 1, count, dtype, np.sqrt(2.0))
    inp = synth.make_swiglu_inputs(cfg, seed=count)
    h = ffn.ffn_swiglu(to_dev(inp["gate"], dtype), to_dev(inp["up"], dtype))
    ref = oracle_lib.swiglu(widen(inp["gate"], dtype), widen(inp["up"], dtype))
    assert_rounded(to_host64(h), ref, dtype)


def test_swiglu_special_values_and_in_place(ffn):
    import torch
    gate = torch.tensor([0.0, -100.0, -1e4, 30.0, 1.0986123, 5.0, -3.0, 2.0], device="cuda")
    up = torch.tensor([3.0, 2.0, 1.0, 1.0, 2.0, 0.0, -1.0, 1.0], device="cuda")
    h = ffn.ffn_swiglu(gate, up)
    ref = np.array([0.0, 0.0, 0.0, 30.0, 1.5 * 1.0986123, 0.0, 3.0 / (1 + np.exp(3.0)), 2.0 / (1 + np.exp(-2.0))])
    got = h.cpu().numpy()
    assert np.all(np.isfinite(got))
    assert np.allclose(got, ref, rtol=1e-5, atol=1e-7)
    ffn.ffn_swiglu(gate, up, out=gate)  # in place
    assert np.allclose(gate.cpu().numpy(), ref, rtol=1e-5, atol=1e-7)


def test_swiglu_full_size_fp16(ffn, oracle_lib):
    """Two 16384 x 11008 fp16 tensors ~N(0,2): sampled rows against the oracle."""
    inp = synth.make_swiglu_inputs(synth.C2B_SWIGLU_F16, seed=0)
    h = ffn.ffn_swiglu(to_dev(inp["gate"], "f16"), to_dev(inp["up"], "f16"))
    rows = np.unique(np.concatenate([[0, 16383], np.random.default_rng(1).integers(0, 16384, 40)]))
    ref = oracle_lib.swiglu(widen(inp["gate"][rows], "f16"), widen(inp["up"][rows], "f16"))
    got = to_host64(h[rows])
    assert_lowp(got, ref)              # the bf16 bound, applied to the fp16 workload
    assert_rounded(got, ref, "f16")    # and one fp16 rounding per element


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("d", [8, 520, 4096, 8192])
def test_rmsnorm_many_rows(ffn, oracle_lib, dtype, d):
    """Row counts that take the streaming (shared-memory ring) kernel."""
    cfg = synth.NormConfig("t", 1000, d, 1e-5, dtype)
    inp = synth.make_norm_inputs(cfg, seed=d + 3)
    n = ffn.ffn_rmsnorm(to_dev(inp["x"], dtype), to_dev(inp["g"], dtype), eps=1e-5)
    rows = np.unique(np.concatenate([[0, 303, 304, 999], np.random.default_rng(d).integers(0, 1000, 40)]))
    ref = oracle_lib.rmsnorm(widen(inp["x"][rows], dtype), widen(inp["g"], dtype), 1e-5)
    assert_rounded(to_host64(n[rows]), ref, dtype)


def test_rmsnorm_many_rows_in_place(ffn, oracle_lib):
    inp = synth.make_norm_inputs(synth.C2A_RMSNORM_F16, seed=9, rows=2000, d=1024)
    x = to_dev(inp["x"], "f16")
    ffn.ffn_rmsnorm(x, to_dev(inp["g"], "f16"), eps=1e-5, out=x)
    ref = oracle_lib.rmsnorm(widen(inp["x"], "f16"), widen(inp["g"], "f16"), 1e-5)
    assert_rounded(to_host64(x), ref, "f16")
