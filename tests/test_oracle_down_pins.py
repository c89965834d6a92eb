"""Pins of the oracle's down projection and of the whole expert MLP (no GPU).

The down projection follows page 52 of "@mlx-bun/inference 0.0.0-stage ->
1.0.0", streamed-experts.ts, DOWN_SOURCE: output row h of grouped row p is
the f32 dot product of the packed row h (I/8 words, element k = nibble k % 8
of word k / 8, minus 8) with mid[p], times the f32 row scale of h, rounded
to bf16.  Each test checks the oracle against something other than itself:
exact integer arithmetic (int64 matmul, rational rounding), a float64 BLAS
matmul, a byte-level reading of the packing, closed forms.
"""
from __future__ import annotations

import numpy as np
import pytest

import exact_ref as X
from up_swiglu_gb300 import synthetic as syn


def _pack(wq: np.ndarray) -> np.ndarray:
    """Integer weights 0..15 [..., K] -> uint32 words [..., K/8] (element k
    in word k // 8 at bits 4 * (k % 8))."""
    *lead, K = wq.shape
    w = wq.reshape(*lead, K // 8, 8).astype(np.uint64)
    word = np.zeros((*lead, K // 8), dtype=np.uint64)
    for p in range(8):
        word |= w[..., p] << np.uint64(4 * p)
    return word.astype(np.uint32)


def _offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def _expert_of_rows(offs):
    return np.repeat(np.arange(len(offs) - 1), np.diff(offs))


def _bf16_of(v: float) -> int:
    return X.bf16_bits(X.round_bf16(X.round_f32(v)))


@pytest.mark.parametrize("counts,I,H", [([1], 8, 16), ([2, 0, 3], 16, 40),
                                        ([5, 1], 64, 24), ([0, 4], 1536, 32)])
def test_down_exact_integer_brute_force(oracle_mod, counts, I, H):
    """Integer mid in [-8, 8] and power-of-two scales: D is an exact integer
    (int64 matmul), out32 = D * s exactly, out its bf16 rounding (exact
    rational rounding).  H != I everywhere, so a transposed weight matrix or
    an index slip cannot pass."""
    rng = np.random.default_rng(100 + I + H)
    E, M = len(counts), int(sum(counts))
    wq = rng.integers(0, 16, size=(E, H, I))
    midi = rng.integers(-8, 9, size=(M, I))
    ds = np.ldexp(np.float32(1), -rng.integers(0, 8, size=(E, H))).astype(
        np.float32)
    offs = _offsets(counts)
    mid = syn.f32_to_bf16_bits(midi.astype(np.float32))
    d = oracle_mod.down_proj(mid, _pack(wq), ds, offs, want_debug=True)
    eo = _expert_of_rows(offs)
    for p in range(M):
        D = (wq[eo[p]] - 8) @ midi[p]                     # int64, exact
        want32 = (D * ds[eo[p]].astype(np.float64)).astype(np.float32)
        assert np.array_equal(d["out32"][p], want32), p
        for h in range(H):
            assert d["out"][p, h] == _bf16_of(float(want32[h])), (p, h)
        assert np.array_equal(d["dabs"][p],
                              (np.abs(wq[eo[p]] - 8) @ np.abs(midi[p]))
                              .astype(np.float64))


def test_down_one_hot_reads_the_packed_byte(oracle_mod):
    """mid = the unit vector at k: out[h] reads weight (h, k) alone.  The
    expected nibble is read from the little-endian bytes of the words (byte
    k // 2 of the row, low nibble for even k), not through the packing rule
    the oracle itself uses."""
    E, H, I = 1, 24, 64
    dw = syn.words_u32(9, syn.S_DOWN_W, E * H * I // 8).reshape(E, H, I // 8)
    ds = (0.5 + syn.uniform(9, syn.S_DOWN_S, E * H)).astype(
        np.float32).reshape(E, H)
    rows = dw.view(np.uint8).reshape(E, H, I // 2)
    one = syn.f32_to_bf16_bits(np.array([1.0], np.float32))[0]
    for k in (0, 1, 7, 8, 9, 31, 62, 63):
        mid = np.zeros((1, I), np.uint16)
        mid[0, k] = one
        d = oracle_mod.down_proj(mid, dw, ds, [0, 1], want_debug=True)
        b = rows[0, :, k // 2].astype(np.int64)
        nib = (b & 0xF) if k % 2 == 0 else (b >> 4)
        want32 = ((nib - 8) * ds[0].astype(np.float64)).astype(np.float32)
        assert np.array_equal(d["out32"][0], want32), k


def test_down_float64_matmul_cross_check(oracle_mod):
    """Real-valued mid: the oracle's f32 value before rounding is the f32
    rounding of a float64 BLAS matmul of the dense dequantised weights times
    the scale (within one f32 ulp: the two f64 sums differ in order only),
    and dabs = |W| @ |mid|."""
    E, H, I = 2, 48, 1024
    counts = [3, 2]
    dw = syn.words_u32(13, syn.S_DOWN_W, E * H * I // 8).reshape(E, H, I // 8)
    ds = (0.002 + 0.018 * syn.uniform(13, syn.S_DOWN_S, E * H)).astype(
        np.float32).reshape(E, H)
    mid = syn.normal_x(13, sum(counts), I, std=0.3)
    k = np.arange(I)
    W = ((dw[:, :, k // 8] >> (4 * (k % 8)).astype(np.uint32)) & 0xF)\
        .astype(np.float64) - 8.0
    mf = syn.bf16_bits_to_f32(mid).astype(np.float64)
    offs = _offsets(counts)
    d = oracle_mod.down_proj(mid, dw, ds, offs, want_debug=True)
    eo = _expert_of_rows(offs)
    for p in range(sum(counts)):
        D = W[eo[p]] @ mf[p]
        want = (D * ds[eo[p]].astype(np.float64)).astype(np.float32)
        assert np.all(np.abs(d["out32"][p] - want)
                      <= np.abs(want) * 2.0 ** -23 + 1e-30)
        assert np.allclose(d["dabs"][p], np.abs(W[eo[p]]) @ np.abs(mf[p]),
                           rtol=1e-13)


def test_down_closed_forms_and_expert_choice(oracle_mod):
    """Every nibble 8: out = +0.  Expert e with every nibble 9 + e (weight
    e + 1) and scale 2^-3: out[p][h] = bf16((e + 1) * sum(mid[p]) / 8), so a
    row read with another expert's weights fails."""
    E, H, I = 3, 16, 256
    counts = [2, 1, 3]
    offs = _offsets(counts)
    mid = syn.normal_x(17, sum(counts), I)
    z = oracle_mod.down_proj(mid, np.full((E, H, I // 8), 0x88888888,
                                          np.uint32),
                             np.ones((E, H), np.float32), offs)
    assert np.all(z == 0)
    words = np.stack([np.full((H, I // 8), int("9ABCDEF0"[e] * 8, 16),
                              np.uint32) for e in range(E)])
    d = oracle_mod.down_proj(mid, words, np.full((E, H), 0.125, np.float32),
                             offs)
    mf = syn.bf16_bits_to_f32(mid).astype(np.float64)
    eo = _expert_of_rows(offs)
    for p in range(sum(counts)):
        want = _bf16_of(float((eo[p] + 1) * np.sum(mf[p]) * 0.125))
        assert np.all(d[p] == want), p


def test_down_sampled_equals_full_and_rejects_bad_arguments(oracle_mod):
    E, H, I = 3, 40, 128
    counts = [2, 0, 3]
    offs = _offsets(counts)
    dw = syn.words_u32(21, syn.S_DOWN_W, E * H * I // 8).reshape(E, H, I // 8)
    ds = (0.01 * (1 + syn.uniform(21, syn.S_DOWN_S, E * H))).astype(
        np.float32).reshape(E, H)
    mid = syn.normal_x(21, 5, I)
    full = oracle_mod.down_proj(mid, dw, ds, offs, want_debug=True)
    rows, cols = np.array([0, 4, 2, 2, 1]), np.array([39, 0, 17, 18, 5])
    s = oracle_mod.down_proj_sampled(mid, dw, ds, offs, rows, cols)
    assert np.array_equal(s["out"], full["out"][rows, cols])
    assert np.array_equal(s["out32"], full["out32"][rows, cols])
    with pytest.raises(ValueError):           # offsets end below M
        oracle_mod.down_proj(mid, dw, ds, [0, 1, 2, 4])
    with pytest.raises(ValueError):           # I not a multiple of 8
        oracle_mod.down_proj(mid[:, :12], dw[:, :, :1], ds, offs)
    with pytest.raises(ValueError):           # sampled column past H
        oracle_mod.down_proj_sampled(mid, dw, ds, offs, [0], [H])


def test_expert_mlp_is_gate_up_then_down(oracle_mod):
    """The MLP's mid is the gate/up output (pinned elsewhere); with every
    down nibble 9 and unit scales its output is bf16(sum_i mid[p][i]) for
    every h (closed form, float64 sum, exact rounding)."""
    E, I, H, T, k = 3, 64, 128, 4, 2
    x = syn.normal_x(23, T, H)
    gw, uw, gs, us = syn.weights(23, E, I, H)
    offs, tok, _ = oracle_mod.group_rows(syn.route_uniform(23, T, k, E), E)
    dw = np.full((E, H, I // 8), 0x99999999, np.uint32)
    mid, out = oracle_mod.expert_mlp(x, gw, uw, gs, us, dw,
                                     np.ones((E, H), np.float32), offs, tok)
    assert np.array_equal(mid, oracle_mod.gate_up_swiglu(x, gw, uw, gs, us,
                                                         offs, tok))
    mf = syn.bf16_bits_to_f32(mid).astype(np.float64)
    for p in range(T * k):
        assert np.all(out[p] == _bf16_of(float(np.sum(mf[p])))), p
