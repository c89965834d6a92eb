"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks the oracle against what the pages and the mathematics fix:
hand-derived tables (tests/golden/), exact rational arithmetic, a 300-bit
exponential, exact integer brute force, a float64 library matmul, closed
forms and invariants.  Page citations are to "@mlx-bun/inference
0.0.0-stage -> 1.0.0": page 52 streamed-experts.ts GATE_UP_SOURCE (the row
arithmetic and the tail), page 54 codebook.ts trellis_bf16 (the rounding).
"""
from __future__ import annotations

import math
import os
import random
from fractions import Fraction

import numpy as np
import pytest

import exact_ref as X
from up_swiglu_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


def _pack(wq: np.ndarray) -> np.ndarray:
    """Pack integer weights in 0..15 [..., H] into uint32 words [..., H/8]:
    element k goes to word k // 8 at bits 4 * (k % 8) (page 52)."""
    *lead, H = wq.shape
    w = wq.reshape(*lead, H // 8, 8).astype(np.uint64)
    word = np.zeros((*lead, H // 8), dtype=np.uint64)
    for p in range(8):
        word |= w[..., p] << np.uint64(4 * p)
    return word.astype(np.uint32)


# ---------------------------------------------------------------- rounding --

def test_bf16_rne_golden_table(oracle_mod):
    for f32hex, bf16hex, *_ in _read_table("bf16_rne_ties.txt"):
        v = X.f32_from_bits(int(f32hex, 16))
        assert oracle_mod.bf16_rne(v) == int(bf16hex, 16), f32hex


def test_bf16_rne_matches_exact_rounding_random(oracle_mod):
    rng = random.Random(7)
    for _ in range(20000):
        b = rng.getrandbits(32)
        if (b >> 23) & 0xFF == 0xFF:
            continue
        v = X.f32_from_bits(b)
        want = X.bf16_bits(X.round_bf16(v))
        assert oracle_mod.bf16_rne(v) == want, hex(b)


# ------------------------------------------------------------------- tail --

def test_tail_exhaustive_against_exact_chain(oracle_mod):
    """All 65,536 bf16 gate values: sigmoidT and siluT equal the exact f32
    chain (300-bit exp, rational roundings)."""
    sig, silu = X.exact_tail_tables()
    bad = []
    for b in range(65536):
        if sig[b] < 0:
            continue
        r = oracle_mod.tail(X.bf16_value(b), 1.0)
        if r[0] != b or r[2] != sig[b] or r[3] != silu[b]:
            bad.append(b)
    assert not bad, [hex(b) for b in bad[:10]]


def test_tail_closed_forms(oracle_mod):
    # sigmoid(0) = 1/2 exactly: silu(0) = +0, and out = +0 for any up
    assert oracle_mod.tail(0.0, 3.0) == (0x0000, 0x4040, 0x3F00, 0x0000,
                                         0x0000)
    # g >= 8: 1 - sigmoid(g) < 2^-9, sigmoidT = 1, siluT = gateT
    for g in (8.0, 30.0, 1000.0, 3.0e38):
        gT, _, sT, siluT, _ = oracle_mod.tail(g, 1.0)
        assert sT == 0x3F80 and siluT == gT
    # exp(-g) overflows f32 for g <= -89: sigmoid = +0, siluT = -0
    for g in (-89.0, -100.0, -3.0e38):
        _, _, sT, siluT, out = oracle_mod.tail(g, 2.0)
        assert sT == 0x0000 and siluT == 0x8000 and out == 0x8000
    # g = -88: sigmoid lands in the f32 subnormal range and is kept
    s32 = X.exact_sigmoid_f32_chain(-88.0)
    assert 0 < s32 < 2.0 ** -126
    assert oracle_mod.tail(-88.0, 1.0)[2] == X.bf16_bits(X.round_bf16(s32))
    # the tail is odd in up: out(g, -u) = -out(g, u)
    for g, u in ((1.5, 2.25), (-3.0, 0.75), (0.125, -7.0)):
        assert oracle_mod.tail(g, -u)[4] == oracle_mod.tail(g, u)[4] ^ 0x8000


def test_tail_sigmoid_rounding_matters(oracle_mod):
    """The page rounds the sigmoid to bf16 before the silu product; the
    'sigmoid in f32' reading differs for some inputs (so the flag is live)."""
    diff = 0
    for b in range(0x3C00, 0x4200):
        g = X.bf16_value(b)
        if oracle_mod.tail(g, 1.0, 0)[3] != oracle_mod.tail(g, 1.0, 1)[3]:
            diff += 1
    assert diff > 0


def test_tail_f32_sigmoid_reading_exhaustive(oracle_mod):
    """The oracle's alternative reading (silu_mode 1: the sigmoid kept in
    f32 for the silu product) on all 65,536 bf16 gate values against the
    exact chain: 300-bit exp, every step rounded by rational arithmetic,
    siluT = bf16(RN32(gateT * s32)); and out = bf16(siluT * upT) for two
    up values, one of them negative."""
    sig, silu = X.exact_tail_tables_f32_sigmoid()
    keep = np.nonzero(sig >= 0)[0]
    g = np.array([X.bf16_value(int(b)) for b in keep], np.float32)
    for up in (1.0, -2.75):
        r = oracle_mod.tail_array(g, np.full_like(g, up), silu_mode=1)
        assert np.array_equal(r[:, 0], keep.astype(np.uint16))
        assert np.array_equal(r[:, 2], sig[keep].astype(np.uint16))
        bad = np.nonzero(r[:, 3] != silu[keep].astype(np.uint16))[0]
        assert bad.size == 0, [hex(int(keep[i])) for i in bad[:10]]
        uT = X.round_bf16(up)
        want = np.array([X.bf16_bits(X.round_bf16(X.mul_f32(
            X.bf16_value(int(s)), uT))) for s in silu[keep]], np.uint16)
        assert np.array_equal(r[:, 4], want)


# -------------------------------------------------- worked example (golden) --

def test_worked_example(oracle_mod):
    kv = {r[0]: r[1:] for r in _read_table("worked_example.txt")}
    H = int(kv["H"][0])
    x = np.array([float(v) for v in kv["x"]], np.float32)
    xb = syn.f32_to_bf16_bits(x).reshape(1, H)
    gw = np.array([[[int(kv["gate_word"][0], 16)]]], np.uint32)
    uw = np.array([[[int(kv["up_word"][0], 16)]]], np.uint32)
    gs = np.array([[float(kv["gate_scale"][0])]], np.float32)
    us = np.array([[float(kv["up_scale"][0])]], np.float32)
    d = oracle_mod.gate_up_swiglu(xb, gw, uw, gs, us, [0, 1], [0],
                                  want_debug=True)
    assert d["gdot"][0, 0] == float(kv["G"][0])
    assert d["udot"][0, 0] == float(kv["U"][0])
    assert d["gate32"][0, 0] == float(kv["gate32"][0])
    assert d["up32"][0, 0] == float(kv["up32"][0])
    gT, uT, sT, siluT, out = oracle_mod.tail(d["gate32"][0, 0],
                                             d["up32"][0, 0])
    assert (gT, uT, sT, siluT) == tuple(
        int(kv[k][0], 16) for k in ("gateT", "upT", "sigmoidT", "siluT"))
    assert out == int(kv["out"][0], 16) == d["out"][0, 0]


# ------------------------------------------------ exact integer brute force --

def _exact_case(rng, E, I, H, T, k):
    wq_g = rng.integers(0, 16, size=(E, I, H))
    wq_u = rng.integers(0, 16, size=(E, I, H))
    xi = rng.integers(-8, 9, size=(T, H))
    gs = np.ldexp(np.float32(1), -rng.integers(4, 10, size=(E, I))).astype(
        np.float32)
    us = np.ldexp(np.float32(1), -rng.integers(4, 10, size=(E, I))).astype(
        np.float32)
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(
        np.int32)
    return wq_g, wq_u, xi, gs, us, topk


@pytest.mark.parametrize("E,I,H,T,k", [(1, 4, 8, 1, 1), (3, 8, 64, 5, 2),
                                       (4, 12, 5120, 3, 3)])
def test_exact_integer_brute_force(oracle_mod, E, I, H, T, k):
    """Integer activations in [-8, 8], power-of-two scales: G and U are exact
    integers (int64 matmul here), gate32 = G * scale exactly, and the output
    is the exact tail of those values."""
    rng = np.random.default_rng(1000 + H)
    wq_g, wq_u, xi, gs, us, topk = _exact_case(rng, E, I, H, T, k)
    xb = syn.f32_to_bf16_bits(xi.astype(np.float32))
    offs, tok, _ = oracle_mod.group_rows(topk, E)
    d = oracle_mod.gate_up_swiglu(xb, _pack(wq_g), _pack(wq_u), gs, us, offs,
                                  tok, want_debug=True)
    M = T * k
    for p in range(M):
        e = int(np.searchsorted(offs, p, side="right") - 1)
        t = tok[p]
        G = (wq_g[e] - 8) @ xi[t]
        U = (wq_u[e] - 8) @ xi[t]
        assert np.array_equal(d["gdot"][p], G.astype(np.float64))
        assert np.array_equal(d["udot"][p], U.astype(np.float64))
        assert np.array_equal(d["gate32"][p], (G * gs[e].astype(np.float64))
                              .astype(np.float32))
        for i in range(I):
            want = X.exact_out_bits(float(G[i] * gs[e, i]),
                                    float(U[i] * us[e, i]))
            assert d["out"][p, i] == want, (p, i)


# ------------------------------------------- float64 matmul cross-check (P4) --

def test_dense_float64_matmul_cross_check(oracle_mod):
    """Real-valued inputs: the oracle's f64 dot products equal a float64
    BLAS matmul of the dequantised dense weights to ~1e-13 of sum|w*x|."""
    E, I, H, T = 2, 16, 1024, 6
    x = syn.normal_x(11, T, H)
    gw, uw, gs, us = syn.weights(11, E, I, H)
    k = np.arange(H)
    # dense dequantisation straight from the page's packing rule
    Wg = ((gw[:, :, k // 8] >> (4 * (k % 8)).astype(np.uint32)) & 0xF)\
        .astype(np.float64) - 8.0
    Wu = ((uw[:, :, k // 8] >> (4 * (k % 8)).astype(np.uint32)) & 0xF)\
        .astype(np.float64) - 8.0
    xf = syn.bf16_bits_to_f32(x).astype(np.float64)
    topk = np.array([[t % E] for t in range(T)], np.int32)
    offs, tok, _ = oracle_mod.group_rows(topk, E)
    d = oracle_mod.gate_up_swiglu(x, gw, uw, gs, us, offs, tok,
                                  want_debug=True)
    for p in range(T):
        e = int(np.searchsorted(offs, p, side="right") - 1)
        t = tok[p]
        G = Wg[e] @ xf[t]
        U = Wu[e] @ xf[t]
        Ga = np.abs(Wg[e]) @ np.abs(xf[t])
        assert np.all(np.abs(d["gdot"][p] - G) <= 1e-13 * Ga)
        assert np.all(np.abs(d["udot"][p] - U) <= 1e-13 * Ga.max() * 4)
        assert np.allclose(d["gabs"][p], Ga, rtol=1e-13)
        want_g32 = (G * gs[e].astype(np.float64)).astype(np.float32)
        assert np.all(np.abs(d["gate32"][p] - want_g32)
                      <= np.abs(want_g32) * 2.0 ** -23 + 1e-30)


# ---------------------------------------------------------- special cases --

def test_special_all_zero_weights(oracle_mod):
    """Every nibble 8 -> every weight 0 -> gate = up = +0 -> out = +0."""
    E, I, H = 2, 8, 64
    x = syn.normal_x(3, 4, H)
    gw = np.full((E, I, H // 8), 0x88888888, np.uint32)
    d = oracle_mod.gate_up_swiglu(x, gw, gw, np.ones((E, I), np.float32),
                                  np.ones((E, I), np.float32), [0, 2, 4],
                                  [0, 1, 2, 3])
    assert np.all(d == 0x0000)


def test_special_one_hot_and_constant_rows(oracle_mod):
    H, I = 128, 16
    x = syn.normal_x(5, 1, H)
    xf = syn.bf16_bits_to_f32(x)[0].astype(np.float64)
    rng = np.random.default_rng(5)
    wq = np.full((1, I, H), 8)
    ks = rng.integers(0, H, size=I)
    vs = rng.integers(0, 16, size=I)
    wq[0, np.arange(I), ks] = vs
    const = rng.integers(0, 16, size=I)
    wc = np.repeat(const[None, :, None], H, axis=2)
    d = oracle_mod.gate_up_swiglu(x, _pack(wq), _pack(wc),
                                  np.ones((1, I), np.float32),
                                  np.ones((1, I), np.float32), [0, 1], [0],
                                  want_debug=True)
    # one-hot row i: G = (v_i - 8) * x[k_i], exactly
    assert np.array_equal(d["gdot"][0], (vs - 8) * xf[ks])
    # constant row: U = (c - 8) * sum(x)
    assert np.allclose(d["udot"][0], (const - 8) * xf.sum(), rtol=1e-14,
                       atol=1e-12)


# ------------------------------------------------------------- invariants --

def test_invariant_token_permutation(oracle_mod):
    E, I, H, T, k = 4, 8, 256, 6, 2
    x = syn.normal_x(21, T, H)
    gw, uw, gs, us = syn.weights(21, E, I, H)
    topk = syn.route_uniform(21, T, k, E)
    offs, tok, _ = oracle_mod.group_rows(topk, E)
    base = oracle_mod.gate_up_swiglu(x, gw, uw, gs, us, offs, tok)
    perm = np.random.default_rng(0).permutation(T)      # new row r = old perm[r]
    inv = np.argsort(perm)
    out = oracle_mod.gate_up_swiglu(x[perm], gw, uw, gs, us, offs, inv[tok])
    assert np.array_equal(out, base)


def test_invariant_expert_relabel_and_batch(oracle_mod):
    """Relabelling experts permutes the row blocks; each row's bits do not
    depend on how many other rows are in the call."""
    E, I, H, T, k = 5, 8, 256, 7, 2
    x = syn.normal_x(22, T, H)
    gw, uw, gs, us = syn.weights(22, E, I, H)
    topk = syn.route_uniform(22, T, k, E)
    offs, tok, rop = oracle_mod.group_rows(topk, E)
    base = oracle_mod.gate_up_swiglu(x, gw, uw, gs, us, offs, tok)
    relabel = np.random.default_rng(1).permutation(E)   # new id = relabel[old]
    order = np.argsort(relabel)                          # old id at new id
    offs2, tok2, rop2 = oracle_mod.group_rows(relabel[topk], E)
    out2 = oracle_mod.gate_up_swiglu(x, gw[order], uw[order], gs[order],
                                     us[order], offs2, tok2)
    assert np.array_equal(out2[rop2], base[rop])
    for e in range(E):                                   # one expert alone
        lo, hi = offs[e], offs[e + 1]
        if hi == lo:
            continue
        one = oracle_mod.gate_up_swiglu(x, gw[e:e + 1], uw[e:e + 1],
                                        gs[e:e + 1], us[e:e + 1],
                                        [0, hi - lo], tok[lo:hi])
        assert np.array_equal(one, base[lo:hi])


def test_group_rows_is_a_stable_sort(oracle_mod):
    rng = np.random.default_rng(3)
    for T, k, E in ((1, 1, 1), (9, 3, 4), (50, 8, 16), (64, 8, 160)):
        topk = rng.integers(0, E, size=(T, k)).astype(np.int32)
        offs, tok, rop = oracle_mod.group_rows(topk, E)
        pairs = sorted(range(T * k), key=lambda q: topk.flat[q])  # stable
        assert list(tok) == [q // k for q in pairs]
        assert list(rop[pairs]) == list(range(T * k))
        counts = np.bincount(topk.ravel(), minlength=E)
        assert list(offs) == [0] + list(np.cumsum(counts))
    with pytest.raises(ValueError):
        oracle_mod.group_rows(np.array([[0, 4]], np.int32), 4)


def test_sampled_equals_full(oracle_mod):
    E, I, H, T, k = 3, 16, 512, 5, 2
    x = syn.normal_x(31, T, H)
    gw, uw, gs, us = syn.weights(31, E, I, H)
    offs, tok, _ = oracle_mod.group_rows(syn.route_uniform(31, T, k, E), E)
    full = oracle_mod.gate_up_swiglu(x, gw, uw, gs, us, offs, tok,
                                     want_debug=True)
    rows = np.array([0, 3, 9, 9, 4]), np.array([0, 15, 7, 8, 2])
    s = oracle_mod.gate_up_swiglu_sampled(x, gw, uw, gs, us, offs, tok, *rows)
    assert np.array_equal(s["out"], full["out"][rows])
    assert np.array_equal(s["gate32"], full["gate32"][rows])
    assert np.array_equal(s["gabs"], full["gabs"][rows])


def test_oracle_rejects_inconsistent_arguments(oracle_mod):
    x = syn.normal_x(1, 2, 64)
    gw, uw, gs, us = syn.weights(1, 2, 4, 64)
    with pytest.raises(ValueError):       # offsets do not end at M
        oracle_mod.gate_up_swiglu(x, gw, uw, gs, us, [0, 1, 3], [0, 1])
    with pytest.raises(ValueError):       # token index past T
        oracle_mod.gate_up_swiglu(x, gw, uw, gs, us, [0, 1, 2], [0, 2])
    with pytest.raises(ValueError):       # offsets decrease
        oracle_mod.gate_up_swiglu(x, gw, uw, gs, us, [0, 2, 1], [0])
