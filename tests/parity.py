"""Element-by-element comparison of the CUDA path with the oracle.

Tolerance (derived from the arithmetic; the pages fix no summation order):
  * f32 gate/up before rounding: |g - o| <= 1e-5 * max(|o|, s * A / sqrt(H)),
    where o is the oracle's value, s the row scale and A = sum_k |w_k x_k|.
    s*A/sqrt(H) is the natural size of a dot product of H random-sign terms,
    so the bound is "relative 1e-5" with the denominator floored at that
    size for rows that cancel (an f32 sum in any order errs by about
    2^-24 * sqrt(H) * (partial sums) which stays far below it).
  * the tail is deterministic: given the GPU's own f32 gate/up, its bf16
    output must equal the oracle's tail of those two values, bit for bit.
  * bf16 output vs the oracle's output: equal wherever gateT and upT agree;
    where one of them differs, the oracle's f32 value must lie within the
    f32 tolerance of a bf16 rounding midpoint (the only way a correct f32
    sum can round the other way); those elements are counted and reported.
With integer activations and power-of-two scales every sum is exact, so the
exact mode demands bit equality of out, gate32 and up32.
"""
from __future__ import annotations

import numpy as np

import oracle


def _bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def _near_midpoint(v: np.ndarray, tol: np.ndarray) -> np.ndarray:
    b = _bits(v)
    mid = ((b & np.uint32(0xFFFF0000)) | np.uint32(0x8000)).view(np.float32)
    return np.abs(v.astype(np.float64) - mid.astype(np.float64)) <= tol


def compare(gpu: dict, orc: dict, gs: np.ndarray, us: np.ndarray, H: int,
            exact: bool = False, tail: str = "page") -> dict:
    """gpu: out (uint16), gate32/up32 (f32); orc: out, gate32, up32, gabs,
    uabs; gs/us: per-element row scales.  All arrays share one shape.
    tail: the SwiGLU tail the call ended with ("page" or "mlx").
    Raises AssertionError with a summary on failure; returns statistics."""
    out_g, out_o = gpu["out"], orc["out"]
    assert out_g.shape == out_o.shape
    stats = {"n": int(out_g.size)}
    if exact:
        bad = np.flatnonzero(out_g != out_o)
        assert bad.size == 0, f"exact: {bad.size} outputs differ, first " \
            f"{bad[:5]}: gpu {out_g.ravel()[bad[:5]]} oracle " \
            f"{out_o.ravel()[bad[:5]]}"
        for k in ("gate32", "up32"):
            if k in gpu:
                d = np.flatnonzero(_bits(gpu[k]) != _bits(orc[k]))
                assert d.size == 0, f"exact: {d.size} {k} differ"
        stats["exact"] = True
        return stats

    g, u = gpu["gate32"], gpu["up32"]
    og, ou = orc["gate32"], orc["up32"]
    assert np.all(np.isfinite(g)) and np.all(np.isfinite(u)), "non-finite"
    tg = 1e-5 * np.maximum(np.abs(og).astype(np.float64),
                           gs * orc["gabs"] / np.sqrt(H))
    tu = 1e-5 * np.maximum(np.abs(ou).astype(np.float64),
                           us * orc["uabs"] / np.sqrt(H))
    eg = np.abs(g.astype(np.float64) - og.astype(np.float64))
    eu = np.abs(u.astype(np.float64) - ou.astype(np.float64))
    stats["max_rel_err_gate"] = float(np.max(eg / tg) * 1e-5) if eg.size \
        else 0.0
    stats["max_rel_err_up"] = float(np.max(eu / tu) * 1e-5) if eu.size \
        else 0.0
    vg, vu = np.flatnonzero(eg > tg), np.flatnonzero(eu > tu)
    assert vg.size == 0 and vu.size == 0, \
        f"f32 tolerance: {vg.size} gate and {vu.size} up elements out of " \
        f"1e-5; worst gate err/tol {np.max(eg / tg):.3g}"
    # strict relative-1e-5 violations (reported, not failed: cancellation)
    stats["strict_rel_violations"] = int(
        np.sum(eg > 1e-5 * np.abs(og)) + np.sum(eu > 1e-5 * np.abs(ou)))

    # the tail given the GPU's own f32 values is exact
    tail_of = oracle.tail_mlx_array if tail == "mlx" else oracle.tail_array
    t = tail_of(g.ravel(), u.ravel())
    bad = np.flatnonzero(t[:, 4] != out_g.ravel())
    assert bad.size == 0, f"tail: {bad.size} outputs differ from the " \
        f"oracle tail of the GPU's own gate/up"

    # output vs oracle: equal where the rounded inputs agree
    gT_g, uT_g = t[:, 0], t[:, 1]
    to = tail_of(og.ravel(), ou.ravel())
    gT_o, uT_o = to[:, 0], to[:, 1]
    same = (gT_g == gT_o) & (uT_g == uT_o)
    dif = np.flatnonzero(out_g.ravel() != out_o.ravel())
    assert np.all(same[dif] == False), "equal bf16 inputs, different out"  # noqa: E712
    flipped = np.flatnonzero(~same)
    near = (_near_midpoint(og.ravel()[flipped], tg.ravel()[flipped]) |
            _near_midpoint(ou.ravel()[flipped], tu.ravel()[flipped]))
    assert np.all(near), f"{np.sum(~near)} gateT/upT roundings differ away " \
        f"from a bf16 midpoint"
    stats["midpoint_flips"] = int(flipped.size)
    stats["out_mismatches"] = int(dif.size)
    return stats


def compare_down(gpu: dict, orc: dict, ds: np.ndarray, K: int,
                 exact: bool = False, extra_tol: np.ndarray | None = None
                 ) -> dict:
    """Down projection: gpu out (uint16) and out32 (f32) against the
    oracle's out, out32 and dabs, all [M, H]; ds: the scale of every
    element.  Tolerance as for gate/up: |g - o| <= 1e-5 * max(|o|,
    s * A / sqrt(K)) (+ extra_tol, an f32 allowance for differences in the
    inputs); the bf16 output must be the rounding of the GPU's own f32 value
    and equal the oracle's except where the oracle's f32 value lies within
    the tolerance of a bf16 rounding midpoint.  exact: bit equality."""
    out_g, out_o = gpu["out"], orc["out"]
    assert out_g.shape == out_o.shape
    stats = {"n": int(out_g.size)}
    if exact:
        bad = np.flatnonzero(out_g != out_o)
        assert bad.size == 0, f"exact: {bad.size} outputs differ, first " \
            f"{bad[:5]}: gpu {out_g.ravel()[bad[:5]]} oracle " \
            f"{out_o.ravel()[bad[:5]]}"
        if "out32" in gpu:
            d = np.flatnonzero(_bits(gpu["out32"]) != _bits(orc["out32"]))
            assert d.size == 0, f"exact: {d.size} out32 differ"
        stats["exact"] = True
        return stats
    g, o = gpu["out32"], orc["out32"]
    assert np.all(np.isfinite(g)), "non-finite"
    tol = 1e-5 * np.maximum(np.abs(o).astype(np.float64),
                            ds * orc["dabs"] / np.sqrt(K))
    if extra_tol is not None:
        tol = tol + extra_tol
    err = np.abs(g.astype(np.float64) - o.astype(np.float64))
    viol = np.flatnonzero(err > tol)
    assert viol.size == 0, f"f32 tolerance: {viol.size} elements out; " \
        f"worst err/tol {np.max(err / tol):.3g}"
    stats["max_err_over_tol"] = float(np.max(err / tol)) if err.size else 0.0
    # the rounding of the GPU's own f32 value
    own = oracle.bf16_rne_array(g.ravel())
    assert np.array_equal(own, out_g.ravel()), "out is not bf16(out32)"
    dif = np.flatnonzero(out_g.ravel() != out_o.ravel())
    near = _near_midpoint(o.ravel()[dif], tol.ravel()[dif])
    if extra_tol is None:
        assert np.all(near), f"{np.sum(~near)} outputs differ away from a " \
            f"bf16 midpoint"
    stats["out_mismatches"] = int(dif.size)
    return stats


def mid_flip_allowance(orc: dict, gs: np.ndarray, us: np.ndarray, H: int
                       ) -> np.ndarray:
    """For each intermediate element: the largest change of the bf16 mid
    that a correct f32 gate/up can cause, from the oracle alone (orc: the
    gate/up oracle's gate32, up32, gabs, uabs).  Where the oracle's gate32
    (up32) lies within the gate/up f32 tolerance of a bf16 midpoint, both
    neighbouring bf16 values are possible; the oracle's tail of every
    possible (gateT, upT) pair bounds the change.  Returns f64 of the same
    shape (zero where no rounding can flip)."""
    g, u = orc["gate32"], orc["up32"]
    tg = 1e-5 * np.maximum(np.abs(g).astype(np.float64),
                           gs * orc["gabs"] / np.sqrt(H))
    tu = 1e-5 * np.maximum(np.abs(u).astype(np.float64),
                           us * orc["uabs"] / np.sqrt(H))
    fg = _near_midpoint(g, tg).ravel()
    fu = _near_midpoint(u, tu).ravel()

    def value(bits):
        return (bits.astype(np.uint32) << 16).view(np.float32) \
            .astype(np.float64)

    base = value(oracle.tail_array(g.ravel(), u.ravel())[:, 4])

    def cands(v, flip):
        b = _bits(v).ravel() & np.uint32(0xFFFF0000)
        lo = b.view(np.float32)
        hi = (b + np.uint32(0x10000)).view(np.float32)
        return [np.where(flip, lo, v.ravel()), np.where(flip, hi, v.ravel())]

    out = np.zeros(g.size, np.float64)
    for gc in cands(g, fg):
        for uc in cands(u, fu):
            t = value(oracle.tail_array(gc, uc)[:, 4])
            out = np.maximum(out, np.abs(t - base))
    return out.reshape(g.shape)


def _ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (the smallest subnormal spacing at 0)."""
    a = np.abs(np.asarray(v, np.float64))
    _, e = np.frexp(a)
    return np.where(a > 0, np.maximum(np.ldexp(1.0, e - 8), 2.0 ** -133),
                    2.0 ** -133)


def compare_down_bits(out_g: np.ndarray, orc: dict, ds: np.ndarray, K: int,
                      extra_tol: np.ndarray | None = None) -> dict:
    """Down outputs known only as bf16 (the fused MLP call): each must lie
    within the f32 tolerance (+ extra_tol) plus half a bf16 spacing of the
    oracle's f32 value (the rounding of a value inside the tolerance)."""
    o = orc["out32"].astype(np.float64)
    tol = 1e-5 * np.maximum(np.abs(o), ds * orc["dabs"] / np.sqrt(K))
    if extra_tol is not None:
        tol = tol + extra_tol
    bound = tol + 0.5 * _ulp_bf16(np.abs(o) + tol)
    g = (out_g.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.all(np.isfinite(g)), "non-finite"
    err = np.abs(g - o)
    viol = np.flatnonzero(err > bound)
    assert viol.size == 0, f"{viol.size} outputs outside the bound; worst " \
        f"err/bound {np.max(err / bound):.3g}"
    return {"n": int(out_g.size),
            "out_mismatches": int(np.sum(out_g != orc["out"]))}
