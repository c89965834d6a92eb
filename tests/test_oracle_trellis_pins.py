"""Pins of the oracle's trellis (QTIP 1MAD) gate/up (no GPU).

Pages of "@mlx-bun/inference 0.0.0-stage -> 1.0.0": page 54, trellis/
codebook.ts (the code value of a state and the state of a weight), page 57,
trellis/gate-up-mma.ts and mixed-gate-up-factored.ts (raw code values summed
in f32, the row scale times 1/147.8 applied once per output, gate and up of
possibly different widths).  Each test checks the oracle against something
other than itself: a value worked by hand, a number-theoretic identity, a
shift-register invariant and a Python big-integer reading of the bit stream,
numpy's f16 conversion, exact integer sums."""
from __future__ import annotations

import numpy as np
import pytest

import exact_ref as X
from up_swiglu_gb300 import synthetic as syn


def test_code_value_worked_by_hand(oracle_mod):
    """State 0: x = 76625530 = 4 * 2^24 + 145 * 2^16 + 54 * 2^8 + 122, bytes
    122 + 54 + 145 + 4 = 325, y = 325 - 510 = -185.  State 1: x = 34038481 +
    76625530 = 110664011 = 6 * 2^24 + 152 * 2^16 + 153 * 2^8 + 75, bytes sum
    386, y = -124."""
    assert 4 * 2**24 + 145 * 2**16 + 54 * 2**8 + 122 == 76625530
    assert 6 * 2**24 + 152 * 2**16 + 153 * 2**8 + 75 == 110664011
    assert oracle_mod.trellis_y(0) == -185
    assert oracle_mod.trellis_y(1) == -124


def test_code_values_mod_255_and_range(oracle_mod):
    """The byte sum of x is congruent to x modulo 255 (256 = 1 mod 255), and
    lies in [0, 1020]: checked on every 12-bit state and on random 24-bit
    ones."""
    rng = np.random.default_rng(0)
    states = list(range(4096)) + [int(s) for s in rng.integers(0, 1 << 24,
                                                                2000)]
    for s in states:
        y = oracle_mod.trellis_y(s)
        x = (s * 34038481 + 76625530) % 2**32
        assert 0 <= y + 510 <= 1020, s
        assert (y + 510) % 255 == x % 255, s


@pytest.mark.parametrize("k,L", [(2, 12), (3, 12), (4, 12), (4, 16)])
def test_states_are_a_shift_register_over_the_block(oracle_mod, k, L):
    """State t+1 is state t shifted by k with k fresh bits (its high L - k
    bits are state t's low L - k), and every state equals a window of the
    block's bits read as one Python integer with wrap-around."""
    Tb = 256
    words = syn.words_u32(k + L, 3, Tb * k // 32)
    st, y = oracle_mod.trellis_block(words, Tb, k, L)
    mask = (1 << (L - k)) - 1
    for t in range(Tb - 1):
        assert st[t + 1] >> k == st[t] & mask, t
    nbits = Tb * k
    big = sum(int(w) << (32 * j) for j, w in enumerate(words))
    ring = big | (big << nbits)
    for t in range(Tb):
        p = (Tb - 1 - t) * k
        assert st[t] == (ring >> p) & ((1 << L) - 1), t
        assert y[t] == oracle_mod.trellis_y(int(st[t]))


def test_factored_scale_against_numpy_f16(oracle_mod):
    """RN32(f32(f16 scale) * RN32(1/147.800537109375)), with the f16 value
    converted by numpy, for every finite f16 pattern."""
    rcp = np.float32(1.0 / 147.800537109375)
    bits = np.arange(65536, dtype=np.uint16)
    vals = bits.view(np.float16).astype(np.float32)
    fin = np.isfinite(vals)
    with np.errstate(invalid="ignore"):
        want = (vals * rcp).astype(np.float32)
    for b in bits[fin][::97]:
        got = np.float32(oracle_mod.trellis_scale(int(b)))
        assert got == want[b] or (got == 0 and want[b] == 0), hex(b)


def _decode_rows(oracle_mod, codes, H, Tb, k, L):
    """y [rows, H] of rows of codes (each row H / Tb blocks)."""
    rows = codes.reshape(-1, codes.shape[-1])
    wpb = Tb * k // 32
    out = np.zeros((rows.shape[0], H), np.int64)
    for r in range(rows.shape[0]):
        for b in range(H // Tb):
            _, y = oracle_mod.trellis_block(rows[r, b * wpb:(b + 1) * wpb],
                                            Tb, k, L)
            out[r, b * Tb:(b + 1) * Tb] = y
    return out.reshape(*codes.shape[:-1], H)


@pytest.mark.parametrize("kg,ku,tail", [(4, 4, "page"), (2, 4, "page"),
                                        (3, 2, "page"), (4, 3, "mlx"),
                                        (2, 2, "mlx")])
def test_gate_up_exact_integer_brute_force(oracle_mod, kg, ku, tail):
    """Integer activations in [-2, 2]: G and U are exact integers (int64
    matmul of the decoded code values), gate32 = RN32(G * scale) with the
    factored scale formed in numpy float32, and the output is the exact
    tail (page 52's, or MLX's in bf16 arithmetic); gate and up of different
    widths are decoded each with its own."""
    E, I, H, T, L, Tb = 2, 8, 512, 3, 12, 256
    rng = np.random.default_rng(kg * 10 + ku)
    gc = syn.words_u32(kg, 5, E * I * (H * kg // 32)).reshape(E, I, -1)
    uc = syn.words_u32(ku, 6, E * I * (H * ku // 32)).reshape(E, I, -1)
    gsv = (0.5 + rng.random((E, I))).astype(np.float16)
    usv = (0.5 + rng.random((E, I))).astype(np.float16)
    xi = rng.integers(-2, 3, size=(T, H))
    x = syn.f32_to_bf16_bits(xi.astype(np.float32))
    topk = np.array([[0], [1], [0]], np.int32)
    offs, tok, _ = oracle_mod.group_rows(topk, E)
    d = oracle_mod.trellis_gate_up_swiglu(x, gc, uc, gsv.view(np.uint16),
                                          usv.view(np.uint16), kg, ku, L, Tb,
                                          offs, tok, tail=tail)
    exact_out = X.exact_mlx_out_bits if tail == "mlx" else X.exact_out_bits
    yg = _decode_rows(oracle_mod, gc, H, Tb, kg, L)
    yu = _decode_rows(oracle_mod, uc, H, Tb, ku, L)
    rcp = np.float32(1.0 / 147.800537109375)
    for p in range(T):
        e = int(np.searchsorted(offs, p, side="right") - 1)
        G = yg[e] @ xi[tok[p]]
        U = yu[e] @ xi[tok[p]]
        sg = (gsv[e].astype(np.float32) * rcp).astype(np.float32)
        su = (usv[e].astype(np.float32) * rcp).astype(np.float32)
        g32 = (G * sg.astype(np.float64)).astype(np.float32)
        u32 = (U * su.astype(np.float64)).astype(np.float32)
        assert np.array_equal(d["gate32"][p], g32)
        assert np.array_equal(d["up32"][p], u32)
        for i in range(I):
            assert d["out"][p, i] == exact_out(float(g32[i]),
                                               float(u32[i])), (p, i)


def test_trellis_sampled_equals_full_and_rejects_bad_geometry(oracle_mod):
    E, I, H, T, k, L, Tb = 2, 4, 256, 2, 2, 12, 256
    gc = syn.words_u32(1, 7, E * I * (H * k // 32)).reshape(E, I, -1)
    s = np.full((E, I), 0x3C00, np.uint16)
    x = syn.normal_x(5, T, H)
    offs, tok = np.array([0, 1, 2], np.int32), np.array([0, 1], np.int32)
    full = oracle_mod.trellis_gate_up_swiglu(x, gc, gc, s, s, k, k, L, Tb,
                                             offs, tok)
    r, c = np.array([1, 0, 1]), np.array([3, 0, 2])
    part = oracle_mod.trellis_gate_up_swiglu(x, gc, gc, s, s, k, k, L, Tb,
                                             offs, tok, r, c)
    assert np.array_equal(part["out"], full["out"][r, c])
    with pytest.raises(ValueError):          # H not a multiple of Tb
        oracle_mod.trellis_gate_up_swiglu(x[:, :200], gc, gc, s, s, k, k, L,
                                          Tb, offs, tok)
    with pytest.raises(ValueError):          # Tb * k not whole words
        oracle_mod.trellis_gate_up_swiglu(x, gc, gc, s, s, k, k, L, 24,
                                          offs, tok)
