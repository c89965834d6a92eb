"""Pins of the oracle's Q8 gate/up and down projection (no GPU).

Page 52 of "@mlx-bun/inference 0.0.0-stage -> 1.0.0", streamed-experts.ts,
Q8_GATE_UP_SOURCE and Q8_DOWN_SOURCE: one signed byte per weight, row-major,
no zero point, f32 accumulation, the f32 row scale, then the same bf16
materialisation and SwiGLU tail as Q4.  Each test checks the oracle against
something other than itself (int64 matmul with exact rational rounding, a
byte-level two's-complement reading, a float64 BLAS matmul)."""
from __future__ import annotations

import numpy as np
import pytest

import exact_ref as X
from up_swiglu_gb300 import synthetic as syn


def _offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


@pytest.mark.parametrize("E,I,H,T,k", [(1, 4, 4, 1, 1), (3, 12, 100, 5, 2),
                                       (2, 8, 5120, 3, 2)])
def test_q8_gate_up_exact_integer_brute_force(oracle_mod, E, I, H, T, k):
    """int8 weights over the whole range, integer activations in [-8, 8],
    power-of-two scales: G and U are exact integers (int64 matmul here), the
    f32 values their exact scaled values, the output the exact tail."""
    rng = np.random.default_rng(500 + H)
    wg = rng.integers(-128, 128, size=(E, I, H)).astype(np.int8)
    wu = rng.integers(-128, 128, size=(E, I, H)).astype(np.int8)
    xi = rng.integers(-8, 9, size=(T, H))
    gs = np.ldexp(np.float32(1), -rng.integers(4, 12, size=(E, I))).astype(
        np.float32)
    us = np.ldexp(np.float32(1), -rng.integers(4, 12, size=(E, I))).astype(
        np.float32)
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(
        np.int32)
    offs, tok, _ = oracle_mod.group_rows(topk, E)
    xb = syn.f32_to_bf16_bits(xi.astype(np.float32))
    d = oracle_mod.q8_gate_up_swiglu(xb, wg, wu, gs, us, offs, tok)
    for p in range(T * k):
        e = int(np.searchsorted(offs, p, side="right") - 1)
        G = wg[e].astype(np.int64) @ xi[tok[p]]
        U = wu[e].astype(np.int64) @ xi[tok[p]]
        assert np.array_equal(d["gate32"][p], (G * gs[e].astype(np.float64))
                              .astype(np.float32))
        for i in range(I):
            assert d["out"][p, i] == X.exact_out_bits(
                float(G[i] * gs[e, i]), float(U[i] * us[e, i])), (p, i)


def test_q8_reads_bytes_as_twos_complement(oracle_mod):
    """One-hot activations read single bytes: 0x80 is -128, 0xFF is -1,
    0x7F is 127, 0x01 is 1 (decoded here from the unsigned byte value)."""
    H, I = 8, 4
    raw = np.array([[0x80, 0xFF, 0x7F, 0x01, 0x00, 0xC3, 0x3C, 0x81]] * I,
                   np.uint8)
    raw[1] = raw[1][::-1]
    w = raw.view(np.int8)[None]
    for kx in range(H):
        x = np.zeros((1, H), np.float32)
        x[0, kx] = 1.0
        d = oracle_mod.q8_gate_up_swiglu(syn.f32_to_bf16_bits(x), w, w,
                                         np.ones((1, I), np.float32),
                                         np.ones((1, I), np.float32),
                                         [0, 1], [0])
        want = [b - 256 if b >= 128 else b for b in raw[:, kx].tolist()]
        assert d["gate32"][0].tolist() == [float(v) for v in want], kx


def test_q8_float64_matmul_cross_check(oracle_mod):
    E, I, H, T = 2, 16, 1024, 6
    rng = np.random.default_rng(3)
    wg = rng.integers(-128, 128, size=(E, I, H)).astype(np.int8)
    gs = (0.001 + 0.01 * rng.random((E, I))).astype(np.float32)
    x = syn.normal_x(41, T, H)
    xf = syn.bf16_bits_to_f32(x).astype(np.float64)
    topk = np.array([[t % E] for t in range(T)], np.int32)
    offs, tok, _ = oracle_mod.group_rows(topk, E)
    d = oracle_mod.q8_gate_up_swiglu(x, wg, wg, gs, gs, offs, tok)
    for p in range(T):
        e = int(np.searchsorted(offs, p, side="right") - 1)
        G = wg[e].astype(np.float64) @ xf[tok[p]]
        want = (G * gs[e].astype(np.float64)).astype(np.float32)
        assert np.all(np.abs(d["gate32"][p] - want)
                      <= np.abs(want) * 2.0 ** -23 + 1e-30)
        assert np.allclose(d["gabs"][p],
                           np.abs(wg[e].astype(np.float64)) @ np.abs(xf[tok[p]]),
                           rtol=1e-13)


@pytest.mark.parametrize("counts,I,H", [([1], 4, 8), ([3, 0, 2], 64, 24),
                                        ([2, 5], 1536, 40)])
def test_q8_down_exact_integer_brute_force(oracle_mod, counts, I, H):
    rng = np.random.default_rng(700 + I + H)
    E, M = len(counts), int(sum(counts))
    wd = rng.integers(-128, 128, size=(E, H, I)).astype(np.int8)
    midi = rng.integers(-8, 9, size=(M, I))
    ds = np.ldexp(np.float32(1), -rng.integers(0, 10, size=(E, H))).astype(
        np.float32)
    offs = _offsets(counts)
    d = oracle_mod.q8_down_proj(syn.f32_to_bf16_bits(midi.astype(np.float32)),
                                wd, ds, offs)
    eo = np.repeat(np.arange(E), counts)
    for p in range(M):
        D = wd[eo[p]].astype(np.int64) @ midi[p]
        want32 = (D * ds[eo[p]].astype(np.float64)).astype(np.float32)
        assert np.array_equal(d["out32"][p], want32), p
        for h in range(H):
            assert d["out"][p, h] == X.bf16_bits(
                X.round_bf16(float(want32[h]))), (p, h)


def test_q8_sampled_equals_full_and_rejects_bad_arguments(oracle_mod):
    E, I, H, T, k = 3, 16, 64, 5, 2
    rng = np.random.default_rng(9)
    wg = rng.integers(-128, 128, size=(E, I, H)).astype(np.int8)
    wd = rng.integers(-128, 128, size=(E, H, I)).astype(np.int8)
    sc = (0.01 + 0.01 * rng.random((E, max(I, H)))).astype(np.float32)
    x = syn.normal_x(43, T, H)
    offs, tok, _ = oracle_mod.group_rows(syn.route_uniform(43, T, k, E), E)
    full = oracle_mod.q8_gate_up_swiglu(x, wg, wg, sc[:, :I], sc[:, :I],
                                        offs, tok)
    rows, cols = np.array([0, 9, 4, 4]), np.array([15, 0, 3, 4])
    s = oracle_mod.q8_gate_up_swiglu(x, wg, wg, sc[:, :I], sc[:, :I], offs,
                                     tok, rows, cols)
    for key in ("out", "gate32", "gabs"):
        assert np.array_equal(s[key], full[key][rows, cols])
    mid = full["out"]
    fd = oracle_mod.q8_down_proj(mid, wd, sc[:, :H], offs)
    sd = oracle_mod.q8_down_proj(mid, wd, sc[:, :H], offs, rows, cols + 40)
    assert np.array_equal(sd["out"], fd["out"][rows, cols + 40])
    with pytest.raises(ValueError):
        oracle_mod.q8_gate_up_swiglu(x, wg, wg, sc[:, :I], sc[:, :I],
                                     [0, 1, 2, 4], tok)
    with pytest.raises(ValueError):
        oracle_mod.q8_down_proj(mid, wd, sc[:, :H], offs, [0], [H])
