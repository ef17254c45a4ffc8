"""Pins for the float64 oracle: facts fixed by the mathematics, not by the oracle.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when the
oracle disagrees with a closed form, an identity, or a brute-force sum on a
tiny input.  ``tests/test_oracle_pins.py`` runs them on the real oracle;
``tests/test_oracle_mutants.py`` runs them on copies with planted mistakes and
requires that every mistake trips at least one pin.

The pages print no worked numeric example, so the anchors are:
  * RMSNorm ("When to hand-write a GPU kernel on Apple Silicon", Rungs 2 and 4):
    closed form for x=[3,4]; constant rows normalise to sign(c)*g;
    rms(n/g) = sqrt(ms/(ms+eps)); scale invariance; a zero row stays zero.
  * SiLU (same page, Rung 1): silu(0)=0, silu(ln 3) = (3/4) ln 3 since
    sigmoid(ln 3) = 3/4, silu(z) - silu(-z) = z, silu(z)/z = 1/2 + z/4 + O(z^3),
    silu(z) -> z for large z and -> 0 for very negative z.
  * Block: a hand-built case whose projections are closed forms, linearity in
    W_up and W_down, brute force with exactly rounded sums (math.fsum).
  * Q4: dequantised weights equal q*s from the generator's integers and scales,
    element by element; the fp16 decoder matches numpy on all 65536 patterns.
"""

from __future__ import annotations

import math

import numpy as np

import synth

LN3 = math.log(3.0)


def _close(a, b, rtol=1e-13, atol=1e-15):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (a.shape, b.shape)
    err = np.abs(a - b)
    tol = atol + rtol * np.abs(b)
    assert np.all(err <= tol), f"max err {err.max()} (at {np.unravel_index(np.argmax(err - tol), err.shape)})"


# ------------------------------------------------------------------ RMSNorm

def pin_rmsnorm_closed_form(o):
    # x = [3, 4]: mean of squares 12.5, so n = [3, 4] / sqrt(12.5) = [0.6, 0.8]*sqrt(2)
    n = o.rmsnorm([[3.0, 4.0]], [1.0, 1.0], 0.0)
    _close(n, [[0.6 * math.sqrt(2.0), 0.8 * math.sqrt(2.0)]])
    # eps inside the root: sqrt(12.5 + 0.5) = sqrt(13); per-column gain [2, -1]
    n = o.rmsnorm([[3.0, 4.0]], [2.0, -1.0], 0.5)
    _close(n, [[6.0 / math.sqrt(13.0), -4.0 / math.sqrt(13.0)]])
    # a 3-wide row: [1, 2, 2] has mean of squares 3
    n = o.rmsnorm([[1.0, 2.0, 2.0]], [1.0, 0.5, 3.0], 0.0)
    r3 = math.sqrt(3.0)
    _close(n, [[1.0 / r3, 1.0 / r3, 6.0 / r3]])


def pin_rmsnorm_constant_rows(o):
    rng = np.random.default_rng(11)
    d = 7
    g = 1.0 + 0.1 * rng.standard_normal(d)
    for c, eps in ((2.5, 0.0), (-1.25, 0.0), (0.3, 1e-2), (-7.0, 1e-5), (1e-3, 1e-6)):
        n = o.rmsnorm(np.full((1, d), c), g, eps)
        _close(n[0], c / math.sqrt(c * c + eps) * g)


def pin_rmsnorm_unit_rms(o):
    rng = np.random.default_rng(12)
    rows, d = 5, 33
    x = rng.standard_normal((rows, d)) * np.arange(1, rows + 1)[:, None]
    g = 1.0 + 0.1 * rng.standard_normal(d)
    for eps in (0.0, 1e-6, 0.3):
        n = o.rmsnorm(x, g, eps)
        ms = np.array([math.fsum(v * v for v in row) / d for row in x])
        rms = np.sqrt(np.mean((n / g) ** 2, axis=1))
        _close(rms, np.sqrt(ms / (ms + eps)), rtol=1e-12)


def pin_rmsnorm_invariances(o):
    rng = np.random.default_rng(13)
    x = rng.standard_normal((4, 16))
    g = 1.0 + 0.1 * rng.standard_normal(16)
    n = o.rmsnorm(x, g, 0.0)
    _close(o.rmsnorm(3.7 * x, g, 0.0), n, rtol=1e-13)         # scale invariance (eps = 0)
    _close(o.rmsnorm(-x, g, 0.0), -n, rtol=1e-15)             # odd in x
    _close(o.rmsnorm(x, 2.0 * g, 1e-3), 2.0 * o.rmsnorm(x, g, 1e-3), rtol=1e-15)
    perm = rng.permutation(16)                                # column equivariance
    _close(o.rmsnorm(x[:, perm], g[perm], 1e-4), o.rmsnorm(x, g, 1e-4)[:, perm], rtol=1e-13)
    z = o.rmsnorm(np.zeros((2, 16)), g, 1e-6)                 # zero row, eps > 0
    assert np.all(z == 0.0)


# --------------------------------------------------------------------- SiLU

def pin_silu_values(o):
    assert o.silu(0.0) == 0.0
    _close(o.silu(LN3), 0.75 * LN3)                  # sigmoid(ln 3) = 3/4
    _close(o.silu(-LN3), -0.25 * LN3)                # sigmoid(-ln 3) = 1/4
    _close(o.silu(math.log(4.0)), 0.8 * math.log(4.0))
    for z in (0.1, 0.7, 1.3, 2.9, 6.5, 11.0):
        _close(o.silu(z) - o.silu(-z), z, rtol=1e-13, atol=1e-15)
    _close(o.silu(40.0), 40.0, rtol=1e-15)
    v = o.silu(-800.0)                               # exp overflows: the limit is 0
    assert v == 0.0 and not math.isnan(v)
    assert -1e-30 < o.silu(-80.0) < 0.0
    for h in (1e-3, 1e-4):                           # silu(h)/h = 1/2 + h/4 - h^3/48 + ...
        assert abs(o.silu(h) / h - 0.5 - h / 4.0) < h ** 3


def pin_swiglu_values(o):
    gate = np.array([LN3, 0.0, -LN3, 5.0, LN3])
    up = np.array([2.0, 9.0, -4.0, 0.0, -1.0])
    h = o.swiglu(gate, up)
    _close(h, [1.5 * LN3, 0.0, LN3, 0.0, -0.75 * LN3])
    rng = np.random.default_rng(14)
    gq = rng.standard_normal((3, 5)) * 3
    uq = rng.standard_normal((3, 5))
    ref = np.array([[math.fsum([gq[i, j] / (1.0 + math.exp(-gq[i, j]))]) * uq[i, j]
                     for j in range(5)] for i in range(3)])
    _close(o.swiglu(gq, uq), ref, rtol=1e-14)


# ---------------------------------------------------------------- FFN block

def pin_block_closed_form(o):
    """Constant rows with eps = 0 normalise to sign(c)*g = +-1; constant
    projection rows then give G = a_f and U = b_f in closed form."""
    d, F = 4, 3
    x = np.array([[2.5] * d, [-1.5] * d])
    g = np.ones(d)
    a = np.array([LN3, 0.0, -LN3])
    b = np.array([2.0, 5.0, -4.0])
    w_gate = np.repeat(a[:, None] / d, d, axis=1)
    w_up = np.repeat(b[:, None] / d, d, axis=1)
    w_down = np.array([[1.0, 2.0, 3.0], [0.0, -1.0, 4.0], [2.0, 0.0, -2.0], [7.0, 1.0, 1.0]])
    # row 0: n = +1 -> G = a, U = b -> h = [1.5 ln3, 0, ln3]
    # row 1: n = -1 -> G = -a, U = -b -> h = [0.5 ln3, 0, 3 ln3]
    h = np.array([[1.5 * LN3, 0.0, LN3], [0.5 * LN3, 0.0, 3.0 * LN3]])
    expect = h @ w_down.T
    _close(o.ffn_block(x, g, w_gate, w_up, w_down, 0.0), expect, rtol=1e-13, atol=1e-14)


def _brute_block(x, g, wg, wu, wd, eps):
    rows, d = x.shape
    F = wg.shape[0]
    y = np.zeros((rows, d))
    for r in range(rows):
        ms = math.fsum(v * v for v in x[r]) / d
        n = [x[r, c] / math.sqrt(ms + eps) * g[c] for c in range(d)]
        h = []
        for f in range(F):
            G = math.fsum(wg[f, c] * n[c] for c in range(d))
            U = math.fsum(wu[f, c] * n[c] for c in range(d))
            h.append(G / (1.0 + math.exp(-G)) * U)
        for j in range(d):
            y[r, j] = math.fsum(wd[j, f] * h[f] for f in range(F))
    return y


def pin_block_brute_force(o):
    rng = np.random.default_rng(15)
    for rows, d, F, eps in ((1, 2, 3, 1e-6), (3, 5, 7, 1e-5), (2, 8, 4, 0.25)):
        x = rng.standard_normal((rows, d))
        g = 1.0 + 0.1 * rng.standard_normal(d)
        wg = rng.standard_normal((F, d)) / math.sqrt(d)
        wu = rng.standard_normal((F, d)) / math.sqrt(d)
        wd = rng.standard_normal((d, F)) / math.sqrt(F)
        _close(o.ffn_block(x, g, wg, wu, wd, eps), _brute_block(x, g, wg, wu, wd, eps),
               rtol=1e-11, atol=1e-13)


def pin_block_linearity(o):
    rng = np.random.default_rng(16)
    rows, d, F = 3, 6, 10
    x = rng.standard_normal((rows, d))
    g = 1.0 + 0.1 * rng.standard_normal(d)
    wg = rng.standard_normal((F, d))
    wu = rng.standard_normal((F, d))
    wd = rng.standard_normal((d, F))
    y = o.ffn_block(x, g, wg, wu, wd, 1e-6)
    # powers of two scale every product and partial sum exactly
    assert np.array_equal(o.ffn_block(x, g, wg, wu, 2.0 * wd, 1e-6), 2.0 * y)
    assert np.array_equal(o.ffn_block(x, g, wg, 4.0 * wu, wd, 1e-6), 4.0 * y)
    assert np.all(o.ffn_block(x, g, wg, np.zeros_like(wu), wd, 1e-6) == 0.0)
    # constant positive rows (eps = 0) normalise to n = 1; W_gate = 50/d gives
    # G = 50 where sigmoid(50) rounds to 1, so silu is the identity there and
    # y_j = sum_f W_down[j,f] * 50 * sum_c W_up[f,c]
    xc = np.full((2, d), 0.75)
    big = o.ffn_block(xc, np.ones(d), np.full((F, d), 50.0 / d), wu, wd, 0.0)
    U = [math.fsum(wu[f]) for f in range(F)]
    ref = [math.fsum(wd[j, f] * 50.0 * U[f] for f in range(F)) for j in range(d)]
    _close(big, np.array([ref, ref]), rtol=1e-12, atol=1e-12)


def pin_block_rows_independent(o):
    rng = np.random.default_rng(17)
    rows, d, F = 6, 8, 12
    x = rng.standard_normal((rows, d))
    g = 1.0 + 0.1 * rng.standard_normal(d)
    wg, wu = rng.standard_normal((F, d)), rng.standard_normal((F, d))
    wd = rng.standard_normal((d, F))
    full = o.ffn_block(x, g, wg, wu, wd, 1e-5, nthreads=3)
    sub = o.ffn_block(x[[4, 1]], g, wg, wu, wd, 1e-5, nthreads=1)
    assert np.array_equal(sub, full[[4, 1]])


def pin_block_residual(o):
    """The skip connection: with W_down = 0 the block returns x itself; in
    the closed-form block above it adds x row by row to the known output."""
    rng = np.random.default_rng(18)
    rows, d, F = 3, 5, 7
    x = rng.standard_normal((rows, d))
    g = 1.0 + 0.1 * rng.standard_normal(d)
    wg, wu = rng.standard_normal((F, d)), rng.standard_normal((F, d))
    assert np.array_equal(o.ffn_block(x, g, wg, wu, np.zeros((d, F)), 1e-6, residual=True), x)
    d, F = 4, 3
    xc = np.array([[2.5] * d, [-1.5] * d])
    a = np.array([LN3, 0.0, -LN3])
    b = np.array([2.0, 5.0, -4.0])
    w_down = np.array([[1.0, 2.0, 3.0], [0.0, -1.0, 4.0], [2.0, 0.0, -2.0], [7.0, 1.0, 1.0]])
    h = np.array([[1.5 * LN3, 0.0, LN3], [0.5 * LN3, 0.0, 3.0 * LN3]])
    got = o.ffn_block(xc, np.ones(d), np.repeat(a[:, None] / d, d, axis=1), np.repeat(b[:, None] / d, d, axis=1),
                      w_down, 0.0, residual=True)
    _close(got, xc + h @ w_down.T, rtol=1e-13, atol=1e-14)


# ------------------------------------------------------- row sum of squares

def pin_row_sumsq_values(o):
    """Closed forms ([3, 4] -> 25, [1, 2, 2] -> 9, a zero row -> 0), exact
    scaling by powers of two (ss(2^k y) = 4^k ss(y)), and brute force with an
    exactly rounded sum (math.fsum) on random rows of several lengths."""
    _close(o.row_sumsq(np.array([[3.0, 4.0], [0.0, 0.0]])), [25.0, 0.0], rtol=0, atol=0)
    _close(o.row_sumsq(np.array([[1.0, 2.0, 2.0], [-1.0, -2.0, 2.0]])), [9.0, 9.0], rtol=0, atol=0)
    rng = np.random.default_rng(30)
    for d in (1, 7, 64, 333):
        y = rng.standard_normal((5, d))
        ss = o.row_sumsq(y)
        _close(ss, [math.fsum(v * v for v in row) for row in y], rtol=1e-13, atol=0)
        _close(o.row_sumsq(8.0 * y), 64.0 * ss, rtol=0, atol=0)


def pin_row_sumsq_feeds_rmsnorm(o):
    """The statistic is the reduction RMSNorm needs: x / sqrt(ss / d + eps) * g
    is the oracle's own RMSNorm of x, and a row whose every element is c
    gives d * c^2."""
    rng = np.random.default_rng(31)
    rows, d, eps = 4, 48, 1e-5
    x = rng.standard_normal((rows, d))
    g = 1.0 + 0.1 * rng.standard_normal(d)
    ss = o.row_sumsq(x)
    _close(x / np.sqrt(ss / d + eps)[:, None] * g, o.rmsnorm(x, g, eps), rtol=1e-13, atol=1e-15)
    _close(o.row_sumsq(np.full((2, 10), -1.5)), [22.5, 22.5], rtol=0, atol=0)


# ---------------------------------------------------------------------- Q4

def pin_half_decoder(o):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    # decode a spread of patterns (every 7th plus all subnormals and specials)
    pick = np.unique(np.concatenate([np.arange(0, 65536, 7), np.arange(0, 1024),
                                     np.arange(0x8000, 0x8400), [0x7C00, 0xFC00, 0x3C00, 0x7BFF]]))
    for b in pick:
        v = o.half_to_double(int(b))
        r = ref[b]
        if math.isnan(r):
            assert math.isnan(v)
        else:
            assert v == r and math.copysign(1.0, v) == math.copysign(1.0, r), (hex(int(b)), v, r)


def pin_q4_dequant_matches_integers(o):
    rng = np.random.default_rng(18)
    out, inn = 5, 256
    q = rng.integers(-8, 8, size=(out, inn), dtype=np.int8)
    s = (np.abs(rng.standard_normal((out, inn // 32))) / 50.0).astype(np.float16)
    s[0, 0] = np.float16(3e-7)         # a subnormal scale
    qs, sc = synth.pack_q4(q, s)
    w = o.q4_dequant(qs, sc, out, inn)
    ref = q.astype(np.float64) * np.repeat(s.astype(np.float64), 32, axis=1)
    assert np.array_equal(w, ref)


def pin_q4_dequant_partial_groups(o):
    """Rows whose length is not a multiple of 128 (one, two and three
    blocks in the last group): every weight at its own index, the padding
    of the last group never read (it is filled with 0xFF bytes and NaN
    scales here, which would show)."""
    rng = np.random.default_rng(19)
    for inn in (32, 96, 160, 224):
        out = 3
        q = rng.integers(-8, 8, size=(out, inn), dtype=np.int8)
        s = (np.abs(rng.standard_normal((out, inn // 32))) / 40.0).astype(np.float16)
        qs, sc = synth.pack_q4(q, s)
        nb, ngrp = inn // 32, -(-inn // 128)
        assert qs.shape == (out, 64 * ngrp) and sc.shape == (out, 4 * ngrp)
        qs = qs.copy()
        sc = sc.copy()
        g = qs.reshape(out, ngrp, 4, 4, 4)          # [o, G, t, b, e]
        for b in range(nb % 4 or 4, 4):
            g[:, -1, :, b, :] = 0xFF
        sc[:, nb:] = 0x7E00                         # fp16 NaN
        w = o.q4_dequant(qs, sc, out, inn)
        ref = q.astype(np.float64) * np.repeat(s.astype(np.float64), 32, axis=1)
        assert np.array_equal(w, ref), inn


def pin_q4_single_weights(o):
    """One non-zero weight at a time: its value must land at its own index."""
    out, inn = 2, 128
    s = np.ones((out, inn // 32), dtype=np.float16)
    s[1, 2] = np.float16(0.5)
    for o_ in range(out):
        for j in range(inn):
            q = np.zeros((out, inn), dtype=np.int8)
            q[o_, j] = -8 if (j % 3) else 7
            qs, sc = synth.pack_q4(q, s)
            w = o.q4_dequant(qs, sc, out, inn)
            ref = q.astype(np.float64) * np.repeat(s.astype(np.float64), 32, axis=1)
            assert np.array_equal(w, ref), (o_, j)




# --------------------------------------------------------------------- fp8

def pin_e4m3_decoder(o):
    """Every one of the 256 codes against the e4m3 ("fn") conversion of a
    library, plus hand-checked values of the format."""
    import torch
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([o.e4m3_to_double(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    for code, v in ((0x38, 1.0), (0x40, 2.0), (0xB8, -1.0), (0x7E, 448.0), (0x01, 2.0 ** -9),
                    (0x08, 2.0 ** -6), (0x07, 7 * 2.0 ** -9), (0x39, 1.125), (0x00, 0.0)):
        assert o.e4m3_to_double(code) == v, (hex(code), v)
    assert math.isnan(o.e4m3_to_double(0x7F)) and math.isnan(o.e4m3_to_double(0xFF))


def pin_fp8_dequant_rows(o):
    """Each row is its codes' values times that row's scale, nothing else."""
    rng = np.random.default_rng(19)
    out, inn = 5, 24
    codes = rng.integers(0, 256, (out, inn)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C      # no NaN codes
    scales = (rng.standard_normal(out) * 0.01).astype(np.float32)
    w = o.fp8_dequant(codes, scales, out, inn)
    for r in range(out):
        for i in range(inn):
            assert w[r, i] == o.e4m3_to_double(codes[r, i]) * float(scales[r])


def pin_q8_dequant_values(o):
    """Q8_0: every weight is its signed code times its own block's scale,
    checked against numpy's fp16 decoding of the scale bits and the codes'
    integers, with the extreme codes, zero, negative scales and a different
    scale in every block."""
    rng = np.random.default_rng(23)
    out, inn = 3, 128
    q = rng.integers(-128, 128, (out, inn)).astype(np.int8)
    q[0, :4] = [-128, 127, 0, -1]
    scales = (rng.standard_normal((out, inn // 32)) * 0.01).astype(np.float16)
    scales[1, 2] = -0.5
    w = o.q8_dequant(q, scales.view(np.uint16), out, inn)
    ref = q.astype(np.float64) * np.repeat(scales.astype(np.float64), 32, axis=1)
    assert np.array_equal(w, ref)
    assert w[0, 0] == -128.0 * float(scales[0, 0]) and w[0, 1] == 127.0 * float(scales[0, 0])
    assert w[1, 64] == q[1, 64] * -0.5 and w[1, 95] == q[1, 95] * -0.5


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
