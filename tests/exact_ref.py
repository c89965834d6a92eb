"""Exact-arithmetic helpers for pinning the oracle (tests only).

These compute the quantities the oracle approximates by a different route:
rational arithmetic (``fractions.Fraction``) for every rounding, and a
300-bit ``mpmath`` exponential for the sigmoid, so a slip in the oracle's C
(a wrong rounding, a dropped step, a flipped sign) shows up as a mismatch.
Signs of zero follow IEEE-754: a product's sign is the exclusive or of its
factors' signs, and a nonzero value that rounds to zero keeps its sign.
"""
from __future__ import annotations

import functools
import math
import struct
from fractions import Fraction

import numpy as np

_HALF = Fraction(1, 2)


def f32_from_bits(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b & 0xFFFFFFFF))[0]


def f32_bits(v: float) -> int:
    return struct.unpack("<I", struct.pack("<f", v))[0]


def bf16_value(b: int) -> float:
    return f32_from_bits((b & 0xFFFF) << 16)


def is_neg(v: float) -> bool:
    return math.copysign(1.0, v) < 0


def _round(r: Fraction, neg: bool, frac_bits: int) -> float:
    """Round the rational r (whose sign, for r == 0, is ``neg``) to the binary
    format with ``frac_bits`` stored fraction bits and the f32 exponent range
    (f32: 23, bf16: 7): nearest, ties to even, subnormals kept, overflow to
    infinity.  Returns a Python float holding the exact result."""
    sign = -1.0 if (r < 0 or (r == 0 and neg)) else 1.0
    a = abs(r)
    if a == 0:
        return sign * 0.0
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    q = Fraction(2) ** (e - frac_bits)
    n = a / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > _HALF or (rem == _HALF and fl % 2 == 1):
        fl += 1
    v = fl * q
    if v >= Fraction(2) ** 128:
        return sign * math.inf
    return sign * float(v)


def round_f32(v: float) -> float:
    """Exact rounding of a Python float (f64) to f32."""
    if math.isinf(v):
        return v
    return _round(Fraction(v), is_neg(v), 23)


def round_bf16(v: float) -> float:
    """Exact rounding of a Python float to bf16."""
    if math.isinf(v):
        return v
    return _round(Fraction(v), is_neg(v), 7)


def round_f32_frac(r: Fraction, neg: bool = False) -> float:
    return _round(r, neg, 23)


def mul_f32(a: float, b: float) -> float:
    """RN32(a * b) from the exact product."""
    return _round(Fraction(a) * Fraction(b), is_neg(a) != is_neg(b), 23)


def bf16_bits(v: float) -> int:
    """Bits of a value already representable in bf16 (sign of zero kept)."""
    b = f32_bits(v)
    assert b & 0xFFFF == 0, v
    return b >> 16


def exact_sigmoid_f32_chain(g: float) -> float:
    """The page's f32 sigmoid chain with each step correctly rounded:
    s32 = RN32(1 / RN32(1 + RN32(exp(-g)))), exp evaluated to 300 bits."""
    import mpmath
    if -g > 90.0:                 # exp(-g) > 1.2e39: past f32 overflow
        return 0.0                # e32 = +inf, d32 = +inf, 1/inf = +0
    if -g < -104.0:               # exp(-g) < 2^-150: e32 rounds to +0
        e32 = 0.0
    else:
        with mpmath.workprec(300):
            ev = mpmath.exp(mpmath.mpf(-g))
            man, ex = int(ev.man), int(ev.exp)
        r = Fraction(man) * (Fraction(2) ** ex)
        e32 = round_f32_frac(r)
        if math.isinf(e32):
            return 0.0
    d32 = round_f32_frac(Fraction(1) + Fraction(e32))
    return round_f32_frac(Fraction(1) / Fraction(d32))


@functools.lru_cache(maxsize=1)
def exact_sigmoid_f32_table():
    """exact_sigmoid_f32_chain of every finite bf16 gateT pattern b (NaN for
    the non-finite patterns), as f32 values held in Python floats."""
    s32 = [math.nan] * 65536
    for b in range(65536):
        if (b >> 7) & 0xFF == 0xFF:
            continue
        s32[b] = exact_sigmoid_f32_chain(bf16_value(b))
    return s32


@functools.lru_cache(maxsize=1)
def exact_tail_tables():
    """For every finite bf16 gateT pattern b: (sigmoidT bits, siluT bits),
    from the exact chain above.  Non-finite patterns hold -1."""
    sig = np.full(65536, -1, dtype=np.int64)
    silu = np.full(65536, -1, dtype=np.int64)
    s32 = exact_sigmoid_f32_table()
    for b in range(65536):
        if (b >> 7) & 0xFF == 0xFF:
            continue
        g = bf16_value(b)
        sT = round_bf16(s32[b])
        siluT = round_bf16(mul_f32(g, sT))
        sig[b] = bf16_bits(sT)
        silu[b] = bf16_bits(siluT)
    return sig, silu


@functools.lru_cache(maxsize=1)
def exact_tail_tables_f32_sigmoid():
    """The 'sigmoid kept in f32' reading of the tail: for every finite bf16
    gateT pattern b, (sigmoidT bits, siluT bits) with
    siluT = bf16(RN32(gateT * s32)), s32 the exact f32 chain itself (not
    rounded to bf16 first); sigmoidT is still bf16(s32).  Non-finite
    patterns hold -1."""
    sig = np.full(65536, -1, dtype=np.int64)
    silu = np.full(65536, -1, dtype=np.int64)
    s32 = exact_sigmoid_f32_table()
    for b in range(65536):
        if (b >> 7) & 0xFF == 0xFF:
            continue
        g = bf16_value(b)
        sig[b] = bf16_bits(round_bf16(s32[b]))
        silu[b] = bf16_bits(round_bf16(mul_f32(g, s32[b])))
    return sig, silu


def exact_out_bits(gate32: float, up32: float) -> int:
    """Final bf16 output of one element from its f32 gate and up: exact
    roundings plus the exact sigmoid/silu table."""
    gT = round_bf16(gate32)
    uT = round_bf16(up32)
    _, silu = exact_tail_tables()
    siluT = bf16_value(int(silu[bf16_bits(gT)]))
    return bf16_bits(round_bf16(mul_f32(siluT, uT)))


def exact_exp_f32(a: float) -> float:
    """RN32(exp(a)) from a 300-bit exp: +inf past f32 overflow, +0 below the
    f32 subnormal range."""
    import mpmath
    if a > 90.0:                  # exp(a) > 1.2e39
        return math.inf
    if a < -104.0:                # exp(a) < 2^-150
        return 0.0
    with mpmath.workprec(300):
        ev = mpmath.exp(mpmath.mpf(a))
        man, ex = int(ev.man), int(ev.exp)
    return round_f32_frac(Fraction(man) * (Fraction(2) ** ex))


def exact_mlx_sigmoid_bf16(g: float) -> float:
    """Sigmoid of MLX's compiled SwiGLU in bf16 arithmetic: every step's
    exact result rounded to f32 and then to bf16; 1 / (1 + exp(|g|)) for
    negative g (not for -0), one minus it otherwise."""
    e = round_bf16(exact_exp_f32(abs(g)))
    if math.isinf(e):
        y = 0.0
    else:
        d = round_bf16(round_f32_frac(Fraction(1) + Fraction(e)))
        y = round_bf16(round_f32_frac(Fraction(1) / Fraction(d)))
    if g < 0:
        return y
    return round_bf16(round_f32_frac(Fraction(1) - Fraction(y)))


@functools.lru_cache(maxsize=1)
def exact_mlx_tail_tables():
    """For every finite bf16 gateT pattern b: (sigmoidT bits, siluT bits)
    of the MLX tail, from the exact chain above.  Non-finite patterns hold
    -1."""
    sig = np.full(65536, -1, dtype=np.int64)
    silu = np.full(65536, -1, dtype=np.int64)
    for b in range(65536):
        if (b >> 7) & 0xFF == 0xFF:
            continue
        g = bf16_value(b)
        sT = exact_mlx_sigmoid_bf16(g)
        siluT = round_bf16(mul_f32(g, sT))
        sig[b] = bf16_bits(sT)
        silu[b] = bf16_bits(siluT)
    return sig, silu


def exact_mlx_out_bits(gate32: float, up32: float) -> int:
    """Final bf16 output of one element through the MLX tail."""
    gT = round_bf16(gate32)
    uT = round_bf16(up32)
    _, silu = exact_mlx_tail_tables()
    siluT = bf16_value(int(silu[bf16_bits(gT)]))
    return bf16_bits(round_bf16(mul_f32(siluT, uT)))
