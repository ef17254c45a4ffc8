"""Plant plausible mistakes into a copy of the oracle and require the pins to
catch every one of them (CPU only; the mistakes live in temporary copies)."""

import os
import shutil
import subprocess

import pytest

import oracle
import oracle_pins

# (name, exact text in ffn_oracle.c, replacement)
MUTANTS = [
    ("eps_outside_root", "sqrt(ms + c->eps)", "(sqrt(ms) + c->eps)"),
    ("mean_over_d_minus_1", "ss / (double)c->d", "ss / (double)(c->d - 1)"),
    ("abs_instead_of_square", "ss += xr[k] * xr[k];", "ss += fabs(xr[k]);"),
    ("gain_dropped", "nr[k] = xr[k] / root * c->g[k];", "nr[k] = xr[k] / root;"),
    ("gain_wrong_index", "nr[k] = xr[k] / root * c->g[k];", "nr[k] = xr[k] / root * c->g[r % c->d];"),
    ("multiply_by_root", "nr[k] = xr[k] / root * c->g[k];", "nr[k] = xr[k] * root * c->g[k];"),
    ("silu_sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("silu_is_sigmoid", "return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    ("gate_up_swapped", "c->h[i] = oracle_silu(G) * U;", "c->h[i] = oracle_silu(U) * G;"),
    ("up_reads_gate", "const double *wu = c->w_up + f * c->d;", "const double *wu = c->w_gate + f * c->d;"),
    ("down_transposed", "s += wd[f] * hr[f];", "s += c->w_down[(f * c->d + j) % (c->d * c->ffn)] * hr[f];"),
    ("down_drops_last_term", "for (int64_t f = 0; f < c->ffn; ++f) s +=",
     "for (int64_t f = 0; f + 1 < c->ffn; ++f) s +="),
    ("q4_nibbles_swapped", "(j < 16) ? (byte & 0x0F) : (byte >> 4)", "(j < 16) ? (byte >> 4) : (byte & 0x0F)"),
    ("q4_offset_7", "(double)(u - 8) * s", "(double)(u - 7) * s"),
    ("q4_group_not_interleaved", "gp[16 * t + 4 * b + e]", "gp[16 * b + 4 * t + e]"),
    ("q4_row_pitch_unpadded", "const uint8_t *row = qs + o * ngrp * 64;", "const uint8_t *row = qs + o * (in / 2);"),
    ("q4_scale_pitch_unpadded", "scales[o * ngrp * 4 + blk]", "scales[o * nblk + blk]"),
    ("q4_groups_rounded_down", "int64_t ngrp = (in + 127) / 128;", "int64_t ngrp = in / 128;"),
    ("half_bias", "e - 25", "e - 24"),
    ("half_subnormal_scale", "ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    ("e4m3_bias", "ldexp((double)(8 + f), e - 10)", "ldexp((double)(8 + f), e - 11)"),
    ("e4m3_no_implicit_one", "ldexp((double)(8 + f), e - 10)", "ldexp((double)f, e - 7)"),
    ("e4m3_subnormal_scale", "v = ldexp((double)f, -9);", "v = ldexp((double)f, -10);"),
    ("fp8_scale_of_wrong_row", "const double s = (double)scales[o];", "const double s = (double)scales[(o + 1) % out];"),
    ("q8_block_of_16", "scales[o * nblk + i / 32]", "scales[o * nblk + i / 16 % nblk]"),
    ("q8_codes_unsigned", "(double)q[o * in + i] * oracle_half_to_double",
     "(double)(uint8_t)q[o * in + i] * oracle_half_to_double"),
    ("q8_scale_of_next_row", "scales[o * nblk + i / 32]", "scales[((o + 1) % out) * nblk + i / 32]"),
    ("sumsq_abs", "for (int64_t c = 0; c < d; ++c) acc += yr[c] * yr[c];",
     "for (int64_t c = 0; c < d; ++c) acc += fabs(yr[c]);"),
    ("sumsq_mean", "        ss[r] = acc;\n", "        ss[r] = acc / (double)d;\n"),
    ("sumsq_skips_first", "for (int64_t c = 0; c < d; ++c) acc += yr[c] * yr[c];",
     "for (int64_t c = 1; c < d; ++c) acc += yr[c] * yr[c];"),
]


def _failing_pins(o):
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
        except Exception as e:  # a crash also counts as caught
            failed.append(f"{pin.__name__}:{type(e).__name__}")
    return failed


@pytest.fixture(scope="module")
def cc():
    exe = shutil.which("cc") or shutil.which("gcc")
    if not exe:
        pytest.skip("no C compiler")
    return exe


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, cc, name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found in the oracle source"
    mutated = src.replace(old, new)
    path = os.path.join(tmp_path, f"mut_{name}.c")
    with open(path, "w") as f:
        f.write(mutated)
    lib = os.path.join(tmp_path, f"libmut_{name}.so")
    oracle.build(path, lib, cc)
    o = oracle.Oracle(lib, source=path)
    assert _failing_pins(o), f"no pin caught mutant {name}"


def test_unmutated_copy_passes(tmp_path, cc):
    lib = os.path.join(tmp_path, "libcopy.so")
    oracle.build(oracle.SOURCE, lib, cc)
    assert _failing_pins(oracle.Oracle(lib)) == []


def test_compiler_present_for_build():
    assert subprocess.run(["cc", "--version"], capture_output=True).returncode == 0
