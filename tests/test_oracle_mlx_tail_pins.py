"""Pins of the oracle's second SwiGLU tail (no GPU): MLX's compiled SwiGLU
in bf16 arithmetic, the tail of the pages' mixed-width trellis kernel
("@mlx-bun/inference 0.0.0-stage -> 1.0.0", page 57,
trellis/mixed-gate-up-factored.ts; the same sigmoid form appears in the
pages' MLX-style activations).  Reading: every step of the chain is
evaluated in f32 and its result rounded to bf16 before the next step.

Each test checks the oracle against something other than itself: a
300-bit exponential with rational roundings for all 65,536 gate values,
values worked by hand, the limits of the chain."""
from __future__ import annotations

import exact_ref as X


def test_mlx_tail_exhaustive_against_exact_chain(oracle_mod):
    """All finite bf16 gate values: sigmoidT and siluT equal the exact
    chain (300-bit exp, every rounding rational)."""
    sig, silu = X.exact_mlx_tail_tables()
    bad = []
    for b in range(65536):
        if sig[b] < 0:
            continue
        r = oracle_mod.tail_mlx(X.bf16_value(b), 1.0)
        if r[0] != b or r[2] != sig[b] or r[3] != silu[b]:
            bad.append(b)
    assert not bad, [hex(b) for b in bad[:10]]


def test_mlx_tail_worked_by_hand(oracle_mod):
    """g = 1: exp(1) = 2.71828... rounds to bf16 2.71875 (steps of 2^-6 in
    [2, 4)); 1 + 2.71875 = 3.71875 is a bf16 value; 1 / 3.71875 =
    0.268907... rounds to 138 * 2^-9 = 0.26953125; 1 - 0.26953125 =
    0.73046875 = 187 * 2^-8 is a bf16 value: sigmoid 0x3F3B, silu 0x3F3B.
    g = 2: exp(2) = 7.389... -> 7.375 (steps of 2^-5); 8.375 is a bf16
    value; 1 / 8.375 = 0.1194... -> 245 * 2^-11 = 0.11962890625; 1 - that =
    0.88037... -> 225 * 2^-8 = 0.87890625 (0x3F61); silu 1.7578125
    (0x3FE1).  g = -2 takes the other branch: sigmoid 0.11962890625
    (0x3DF5), silu -0.2392578125 (0xBE75)."""
    assert oracle_mod.tail_mlx(1.0, 1.0)[2:4] == (0x3F3B, 0x3F3B)
    assert oracle_mod.tail_mlx(2.0, 1.0)[2:4] == (0x3F61, 0x3FE1)
    assert oracle_mod.tail_mlx(-2.0, 1.0)[2:4] == (0x3DF5, 0xBE75)
    # out = bf16(siluT * upT): 1.7578125 * 3 = 5.2734375 -> 5.28125 (steps
    # of 2^-5 in [4, 8)), 0x40A9
    assert oracle_mod.tail_mlx(2.0, 3.0)[4] == 0x40A9


def test_mlx_tail_limits(oracle_mod):
    # g = 0: exp 1, 1 + 1 = 2, 1/2, 1 - 1/2: sigmoid 1/2, silu +0
    assert oracle_mod.tail_mlx(0.0, 3.0) == (0x0000, 0x4040, 0x3F00, 0x0000,
                                             0x0000)
    # g = -0 is not negative: the same sigmoid, silu -0 * 1/2 = -0
    assert oracle_mod.tail_mlx(-0.0, 3.0) == (0x8000, 0x4040, 0x3F00, 0x8000,
                                              0x8000)
    # g >= 8: 1 / (1 + exp(g)) < 2^-9, 1 minus it rounds to 1: silu = gate
    for g in (8.0, 30.0, 1000.0, 3.0e38):
        gT, _, sT, siluT, _ = oracle_mod.tail_mlx(g, 1.0)
        assert sT == 0x3F80 and siluT == gT
    # exp(|g|) overflows for g <= -89: sigmoid +0, silu -0
    for g in (-89.0, -100.0, -3.0e38):
        _, _, sT, siluT, out = oracle_mod.tail_mlx(g, 2.0)
        assert sT == 0x0000 and siluT == 0x8000 and out == 0x8000
    # g = -88: the sigmoid is a bf16 subnormal and is kept
    s = X.exact_mlx_sigmoid_bf16(-88.0)
    assert 0 < s < 2.0 ** -126
    assert oracle_mod.tail_mlx(-88.0, 1.0)[2] == X.bf16_bits(s)


def test_mlx_tail_branches_are_complements(oracle_mod):
    """For g > 0 the sigmoid is bf16(1 - sigmoid(-g)): the two branches of
    the chain read the same y (catches a swapped branch or a sign slip)."""
    for b in range(0x0001, 0x7F80, 7):
        g = X.bf16_value(b)
        pos = oracle_mod.tail_mlx(g, 1.0)[2]
        neg = oracle_mod.tail_mlx(-g, 1.0)[2]
        want = X.bf16_bits(X.round_bf16(X.round_f32_frac(
            X.Fraction(1) - X.Fraction(X.bf16_value(neg)))))
        assert pos == want, hex(b)


def test_mlx_tail_differs_from_the_page_52_tail(oracle_mod):
    """The two tails round at different points; they disagree on some gate
    values, so the choice between them is live."""
    diff = 0
    for b in range(0x3C00, 0x4200):
        g = X.bf16_value(b)
        if oracle_mod.tail_mlx(g, 1.0)[3] != oracle_mod.tail(g, 1.0)[3]:
            diff += 1
    assert diff > 0


def test_mlx_tail_array_matches_scalar(oracle_mod):
    import numpy as np
    rng = np.random.default_rng(3)
    g = (rng.standard_normal(500) * 6).astype(np.float32)
    u = (rng.standard_normal(500) * 2).astype(np.float32)
    arr = oracle_mod.tail_mlx_array(g, u)
    for j in range(500):
        assert tuple(int(v) for v in arr[j]) == oracle_mod.tail_mlx(
            float(g[j]), float(u[j]))
