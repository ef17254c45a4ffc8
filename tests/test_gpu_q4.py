"""ffn_block_forward_q4 on the GPU against the oracle applied to the same
dequantised weights (the oracle unpacks the packed bytes itself)."""

import numpy as np
import pytest

import synth
from gpu_util import assert_lowp, q4_dev, to_dev, to_host64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ffn():
    from transformer_ffn_rmsnorm_gb300 import ffn as m
    return m


def run_q4(ffn, inp):
    cfg = inp["cfg"]
    return ffn.ffn_block_forward_q4(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"),
                                    q4_dev(inp, "gate"), q4_dev(inp, "up"), q4_dev(inp, "down"),
                                    ffn=cfg.ffn, eps=cfg.eps)


def test_q4_full_size(ffn, oracle_lib):
    """8 rows, d=5120, ffn=17408, Q4 weights."""
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=0)
    assert_lowp(to_host64(run_q4(ffn, inp)), oracle_lib.q4_block_from_inputs(inp))


@pytest.mark.parametrize("rows", [1, 3, 8, 9, 16, 20, 33])
def test_q4_rows(ffn, oracle_lib, rows):
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=rows, rows=rows, d=1024, ffn=2816)
    assert_lowp(to_host64(run_q4(ffn, inp)), oracle_lib.q4_block_from_inputs(inp))


@pytest.mark.parametrize("d,ffn_", [(128, 128), (384, 640), (4096, 2176)])
def test_q4_shapes(ffn, oracle_lib, d, ffn_):
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=d, rows=4, d=d, ffn=ffn_)
    assert_lowp(to_host64(run_q4(ffn, inp)), oracle_lib.q4_block_from_inputs(inp))


def test_q4_single_weight_probe(ffn, oracle_lib):
    """All weights zero except one per matrix: the output isolates one nibble's
    position, scale and sign through the whole path."""
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=1, rows=2, d=256, ffn=256)
    for name, (o, i) in (("gate", (256, 256)), ("up", (256, 256)), ("down", (256, 256))):
        q = np.zeros((o, i), dtype=np.int8)
        if name == "down":
            q[:, :] = np.random.default_rng(3).integers(-8, 8, size=(o, i))
        else:
            q[37, 161] = -7
            q[37, 5] = 6
        s = np.full((o, i // 32), 0.0625, dtype=np.float16)
        inp["q_" + name], inp["s_" + name] = q, s
        inp["qs_" + name], inp["sc_" + name] = synth.pack_q4(q, s)
    y = to_host64(run_q4(ffn, inp))
    ref = oracle_lib.q4_block_from_inputs(inp)
    assert_lowp(y, ref)


def test_q4_deterministic(ffn):
    import hashlib
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=5, rows=8, d=1024, ffn=2048)
    import torch
    hs = {hashlib.sha256(run_q4(ffn, inp).view(torch.int16).cpu().numpy().tobytes()).hexdigest()
          for _ in range(3)}
    assert len(hs) == 1


def test_q4_flags_rejected(ffn):
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=3, rows=2, d=128, ffn=128)
    cfg = inp["cfg"]
    with pytest.raises(ffn.FFNError):
        ffn.ffn_block_forward_q4(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"), q4_dev(inp, "gate"),
                                 q4_dev(inp, "up"), q4_dev(inp, "down"), ffn=cfg.ffn, eps=cfg.eps,
                                 flags=ffn.FFN_ACT_SPLIT)


def test_q4_large_activations(ffn, oracle_lib):
    """Gain x 64 and gate/up block scales x 4 (powers of two, exact): h of
    order 10^4 (up to ~10^5), so the block offsets of n and of h reach ~10^8.
    The streaming kernels carry them as two tf32 terms and take them off
    after the products; the result stays within the bound of the oracle."""
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=71, rows=8, d=1024, ffn=2816)
    gb = inp["g"].astype(np.int32)            # bf16 bit patterns
    exp = (gb >> 7) & 0xFF
    assert np.all((exp > 0) & (exp < 200))    # normal values: x 64 is +6 in the exponent field
    inp["g"] = (gb + (6 << 7)).astype(np.uint16)
    for name in ("gate", "up"):
        inp["s_" + name] = (inp["s_" + name] * np.float16(4)).astype(np.float16)
        inp["qs_" + name], inp["sc_" + name] = synth.pack_q4(inp["q_" + name], inp["s_" + name])
    ref = oracle_lib.q4_block_from_inputs(inp)
    assert_lowp(to_host64(run_q4(ffn, inp)), ref)


@pytest.mark.parametrize("rows", [3, 12])
def test_q4_long_rows(ffn, oracle_lib, rows):
    """d = 16640 (65 stages of 256): the sliced norm kernel writing the
    offset form of the streaming kernels (slices of whole blocks, offsets
    reduced over lane quads); one and two token tiles."""
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=90 + rows, rows=rows, d=16640, ffn=512)
    assert_lowp(to_host64(run_q4(ffn, inp)), oracle_lib.q4_block_from_inputs(inp))


@pytest.mark.parametrize("rows,d,ffn_,residual", [(1, 96, 160, False), (5, 416, 224, True), (12, 32, 96, False),
                                                  (16, 1056, 2080, True)])
def test_q4_partial_groups(ffn, oracle_lib, rows, d, ffn_, residual):
    """d and ffn multiples of 32 but not of 128: rows ending in a padded
    group of 1-3 blocks (the register kernels), one and two token tiles,
    with and without the skip connection."""
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=rows + d, rows=rows, d=d, ffn=ffn_)
    cfg = inp["cfg"]
    y = ffn.ffn_block_forward_q4(to_dev(inp["x"], "bf16"), to_dev(inp["g"], "bf16"), q4_dev(inp, "gate"),
                                 q4_dev(inp, "up"), q4_dev(inp, "down"), ffn=cfg.ffn, eps=cfg.eps,
                                 flags=ffn.FFN_RESIDUAL if residual else 0)
    assert_lowp(to_host64(y), oracle_lib.q4_block_from_inputs(inp, residual=residual))
    ffn.ffn_device_status()
