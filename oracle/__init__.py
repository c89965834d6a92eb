"""CPU oracle for the fused Q4 MoE gate/up + SwiGLU (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py``
may import this package.  The CUDA library never imports, links or calls it,
and it imports nothing from the CUDA library's package.

The arithmetic lives in ``q4moe_oracle.c`` (plain C, f64 accumulation); this
module compiles it with gcc on first use and marshals numpy arrays.  Every
function cites the passage it follows in the C source.  ``group_rows``,
``tail``, ``gate_up_swiglu``, ``down_proj`` and ``expert_mlp`` are pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` (and the ``test_oracle_*_pins.py`` files beside
it for the down projection, Q8, trellis codes and the MLX tail).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libq4moe_oracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_INT = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-fPIC", "-shared", "-Wall", "-Wextra",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.q4o_bf16_rne.restype = ctypes.c_uint16
        lib.q4o_bf16_rne.argtypes = [ctypes.c_float]
        lib.q4o_bf16_to_f32.restype = ctypes.c_float
        lib.q4o_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.q4o_bf16_rne_array.restype = None
        lib.q4o_bf16_rne_array.argtypes = [_I64, _P, _P]
        lib.q4o_tail.restype = None
        lib.q4o_tail.argtypes = [ctypes.c_float, ctypes.c_float, _INT, _P]
        lib.q4o_tail_array.restype = None
        lib.q4o_tail_array.argtypes = [_I64, _P, _P, _INT, _P]
        lib.q4o_gate_up_swiglu.restype = _INT
        lib.q4o_gate_up_swiglu.argtypes = [
            _P, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _P, _P, _I64, _INT,
            _P, _P, _P, _P, _P, _P, _P, _INT]
        lib.q4o_gate_up_swiglu_sampled.restype = _INT
        lib.q4o_gate_up_swiglu_sampled.argtypes = [
            _P, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _P, _P, _I64, _INT,
            _I64, _P, _P, _P, _P, _P, _P, _P, _INT]
        lib.q4o_down_proj.restype = _INT
        lib.q4o_down_proj.argtypes = [
            _P, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _P, _P, _INT]
        lib.q4o_down_proj_sampled.restype = _INT
        lib.q4o_down_proj_sampled.argtypes = [
            _P, _I64, _I64, _I64, _I32, _P, _P, _P, _I64, _P, _P, _P, _P, _P,
            _INT]
        lib.q4o_q8_gate_up_swiglu.restype = _INT
        lib.q4o_q8_gate_up_swiglu.argtypes = [
            _P, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _P, _P, _I64, _INT,
            _I64, _P, _P, _P, _P, _P, _P, _P, _INT]
        lib.q4o_q8_down_proj.restype = _INT
        lib.q4o_q8_down_proj.argtypes = [
            _P, _I64, _I64, _I64, _I32, _P, _P, _P, _I64, _P, _P, _P, _P, _P,
            _INT]
        lib.q4o_trellis_gate_up_swiglu.restype = _INT
        lib.q4o_trellis_gate_up_swiglu.argtypes = [
            _P, _I64, _I64, _I64, _I32, _P, _P, _P, _P, _INT, _INT, _INT,
            _I64, _P, _P, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _INT,
            _INT]
        lib.q4o_tail_mlx.restype = None
        lib.q4o_tail_mlx.argtypes = [ctypes.c_float, ctypes.c_float, _P]
        lib.q4o_tail_mlx_array.restype = None
        lib.q4o_tail_mlx_array.argtypes = [_I64, _P, _P, _P]
        lib.q4o_trellis_y.restype = _INT
        lib.q4o_trellis_y.argtypes = [ctypes.c_uint32]
        lib.q4o_trellis_scale.restype = ctypes.c_float
        lib.q4o_trellis_scale.argtypes = [ctypes.c_uint16]
        lib.q4o_trellis_block_codes.restype = _INT
        lib.q4o_trellis_block_codes.argtypes = [_P, _I64, _INT, _INT, _P]
        lib.q4o_trellis_block_states.restype = _INT
        lib.q4o_trellis_block_states.argtypes = [_P, _I64, _INT, _INT, _P]
        lib.q4o_group_rows.restype = _INT
        lib.q4o_group_rows.argtypes = [_P, _I64, _I32, _I32, _P, _P, _P]
        lib.q4o_max_threads.restype = _INT
        lib.q4o_max_threads.argtypes = []
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_P)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(_load().q4o_max_threads())


def bf16_rne(v: float) -> int:
    """f32 -> bf16 bits, round to nearest even (page 54, trellis_bf16)."""
    return int(_load().q4o_bf16_rne(float(np.float32(v))))


def bf16_rne_array(a) -> np.ndarray:
    flat = _c(np.asarray(a, dtype=np.float32).ravel(), np.float32)
    out = np.zeros(flat.shape[0], np.uint16)
    _load().q4o_bf16_rne_array(flat.shape[0], _ptr(flat), _ptr(out))
    return out.reshape(np.shape(a))


def tail(gate32: float, up32: float, silu_mode: int = 0):
    """(gateT, upT, sigmoidT, siluT, out) bf16 bits for one element
    (page 52, streamed-experts.ts, GATE_UP_SOURCE tail)."""
    res = np.zeros(5, dtype=np.uint16)
    _load().q4o_tail(ctypes.c_float(gate32), ctypes.c_float(up32),
                     int(silu_mode), _ptr(res))
    return tuple(int(v) for v in res)


def tail_mlx(gate32: float, up32: float):
    """(gateT, upT, sigmoidT, siluT, out) bf16 bits for one element through
    MLX's compiled SwiGLU in bf16 arithmetic, the tail of the pages'
    mixed-width trellis kernel (page 57, mixed-gate-up-factored.ts)."""
    res = np.zeros(5, dtype=np.uint16)
    _load().q4o_tail_mlx(ctypes.c_float(gate32), ctypes.c_float(up32),
                         _ptr(res))
    return tuple(int(v) for v in res)


def tail_mlx_array(gate32, up32) -> np.ndarray:
    """tail_mlx() over arrays of f32 gate/up values; uint16 [n, 5]."""
    g = _c(gate32, np.float32).ravel()
    u = _c(up32, np.float32).ravel()
    assert g.shape == u.shape
    res = np.zeros((g.shape[0], 5), dtype=np.uint16)
    _load().q4o_tail_mlx_array(g.shape[0], _ptr(g), _ptr(u), _ptr(res))
    return res


def tail_array(gate32, up32, silu_mode: int = 0) -> np.ndarray:
    """tail() over arrays of f32 gate/up values; returns uint16 [n, 5]."""
    g = _c(gate32, np.float32).ravel()
    u = _c(up32, np.float32).ravel()
    assert g.shape == u.shape
    res = np.zeros((g.shape[0], 5), dtype=np.uint16)
    _load().q4o_tail_array(g.shape[0], _ptr(g), _ptr(u), int(silu_mode),
                           _ptr(res))
    return res


def group_rows(topk_ids, num_experts: int):
    """Stable counting sort of (token, slot) pairs by expert.

    Returns (row_offsets [E+1], token_of_row [T*k], row_of_pair [T*k])."""
    topk = _c(topk_ids, np.int32)
    T, k = topk.shape
    offs = np.zeros(num_experts + 1, dtype=np.int32)
    tok = np.zeros(T * k, dtype=np.int32)
    rop = np.zeros(T * k, dtype=np.int32)
    rc = _load().q4o_group_rows(_ptr(topk), T, k, num_experts, _ptr(offs),
                                _ptr(tok), _ptr(rop))
    if rc != 0:
        raise ValueError(f"oracle group_rows rejected the ids (rc={rc})")
    return offs, tok, rop


def gate_up_swiglu(x_bits, gate_w, up_w, gate_s, up_s, row_offsets,
                   token_of_row, silu_mode: int = 0, nthreads: int = 0,
                   want_debug: bool = False):
    """All M x I outputs of the grouped call.

    x_bits bf16 bits [T, H] (uint16); gate_w/up_w uint32 [E, I, H/8];
    gate_s/up_s f32 [E, I]; row_offsets int32 [E+1]; token_of_row int32 [M].
    Returns out bits [M, I] (uint16), or with want_debug a dict that also
    holds gate32/up32 (f32), gdot/udot (f64 unscaled dots) and gabs/uabs
    (f64 sums of |w*x|)."""
    x = _c(x_bits, np.uint16)
    gw, uw = _c(gate_w, np.uint32), _c(up_w, np.uint32)
    gs, us = _c(gate_s, np.float32), _c(up_s, np.float32)
    offs, tok = _c(row_offsets, np.int32), _c(token_of_row, np.int32)
    T, H = x.shape
    E, I, _ = gw.shape
    M = tok.shape[0]
    out = np.zeros((M, I), dtype=np.uint16)
    dbg = None
    if want_debug:
        dbg = dict(gate32=np.zeros((M, I), np.float32),
                   up32=np.zeros((M, I), np.float32),
                   gdot=np.zeros((M, I), np.float64),
                   udot=np.zeros((M, I), np.float64),
                   gabs=np.zeros((M, I), np.float64),
                   uabs=np.zeros((M, I), np.float64))
    g = (lambda k: _ptr(dbg[k])) if dbg else (lambda k: None)
    rc = _load().q4o_gate_up_swiglu(
        _ptr(x), T, H, I, E, _ptr(gw), _ptr(uw), _ptr(gs), _ptr(us),
        _ptr(offs), _ptr(tok), M, int(silu_mode), _ptr(out), g("gate32"),
        g("up32"), g("gdot"), g("udot"), g("gabs"), g("uabs"), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    if dbg is not None:
        dbg["out"] = out
        return dbg
    return out


def gate_up_swiglu_sampled(x_bits, gate_w, up_w, gate_s, up_s, row_offsets,
                           token_of_row, rows, cols, silu_mode: int = 0,
                           nthreads: int = 0):
    """The outputs at (rows[j], cols[j]) only.  Returns a dict with out (bf16
    bits), gate32/up32 (f32) and gabs/uabs (f64), each of length n."""
    x = _c(x_bits, np.uint16)
    gw, uw = _c(gate_w, np.uint32), _c(up_w, np.uint32)
    gs, us = _c(gate_s, np.float32), _c(up_s, np.float32)
    offs, tok = _c(row_offsets, np.int32), _c(token_of_row, np.int32)
    r, c = _c(rows, np.int64), _c(cols, np.int64)
    T, H = x.shape
    E, I, _ = gw.shape
    n = r.shape[0]
    res = dict(out=np.zeros(n, np.uint16), gate32=np.zeros(n, np.float32),
               up32=np.zeros(n, np.float32), gabs=np.zeros(n, np.float64),
               uabs=np.zeros(n, np.float64))
    rc = _load().q4o_gate_up_swiglu_sampled(
        _ptr(x), T, H, I, E, _ptr(gw), _ptr(uw), _ptr(gs), _ptr(us),
        _ptr(offs), _ptr(tok), tok.shape[0], int(silu_mode), n, _ptr(r),
        _ptr(c), _ptr(res["out"]), _ptr(res["gate32"]), _ptr(res["up32"]),
        _ptr(res["gabs"]), _ptr(res["uabs"]), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return res


def down_proj(mid_bits, down_w, down_s, row_offsets, nthreads: int = 0,
              want_debug: bool = False):
    """All M x H outputs of the grouped down projection (page 52,
    streamed-experts.ts, DOWN_SOURCE).

    mid_bits bf16 bits [M, I] (grouped order); down_w uint32 [E, H, I/8];
    down_s f32 [E, H]; row_offsets int32 [E+1].  Returns out bits [M, H], or
    with want_debug a dict with out, out32 (f32 before the bf16 rounding) and
    dabs (f64 sums of |w*mid|)."""
    mid = _c(mid_bits, np.uint16)
    dw, ds = _c(down_w, np.uint32), _c(down_s, np.float32)
    offs = _c(row_offsets, np.int32)
    M, I = mid.shape
    E, H, _ = dw.shape
    out = np.zeros((M, H), dtype=np.uint16)
    dbg = None
    if want_debug:
        dbg = dict(out32=np.zeros((M, H), np.float32),
                   dabs=np.zeros((M, H), np.float64))
    g = (lambda k: _ptr(dbg[k])) if dbg else (lambda k: None)
    rc = _load().q4o_down_proj(_ptr(mid), M, I, H, E, _ptr(dw), _ptr(ds),
                               _ptr(offs), _ptr(out), g("out32"), g("dabs"),
                               int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    if dbg is not None:
        dbg["out"] = out
        return dbg
    return out


def down_proj_sampled(mid_bits, down_w, down_s, row_offsets, rows, cols,
                      nthreads: int = 0):
    """The down projection at (rows[j], cols[j]) only; mid_bits must hold
    every row that rows names (other rows may be anything).  Returns a dict
    with out (bf16 bits), out32 (f32) and dabs (f64), each of length n."""
    mid = _c(mid_bits, np.uint16)
    dw, ds = _c(down_w, np.uint32), _c(down_s, np.float32)
    offs = _c(row_offsets, np.int32)
    r, c = _c(rows, np.int64), _c(cols, np.int64)
    M, I = mid.shape
    E, H, _ = dw.shape
    n = r.shape[0]
    res = dict(out=np.zeros(n, np.uint16), out32=np.zeros(n, np.float32),
               dabs=np.zeros(n, np.float64))
    rc = _load().q4o_down_proj_sampled(
        _ptr(mid), M, I, H, E, _ptr(dw), _ptr(ds), _ptr(offs), n, _ptr(r),
        _ptr(c), _ptr(res["out"]), _ptr(res["out32"]), _ptr(res["dabs"]),
        int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return res


def expert_mlp(x_bits, gate_w, up_w, gate_s, up_s, down_w, down_s,
               row_offsets, token_of_row, nthreads: int = 0):
    """The whole routed expert MLP as the page runs it (page 52,
    streamed-experts.ts: the gate/up kernel writes mid, the down kernel
    reads it): returns (mid bits [M, I], out bits [M, H])."""
    mid = gate_up_swiglu(x_bits, gate_w, up_w, gate_s, up_s, row_offsets,
                         token_of_row, nthreads=nthreads)
    return mid, down_proj(mid, down_w, down_s, row_offsets,
                          nthreads=nthreads)


def q8_gate_up_swiglu(x_bits, gate_w, up_w, gate_s, up_s, row_offsets,
                      token_of_row, rows=None, cols=None, silu_mode: int = 0,
                      nthreads: int = 0):
    """Q8 gate/up (page 52, Q8_GATE_UP_SOURCE): gate_w/up_w int8 [E, I, H].
    All M x I outputs (arrays [M, I]) or, with rows/cols, those elements
    only (arrays [n]).  Returns a dict with out, gate32, up32, gabs, uabs."""
    x = _c(x_bits, np.uint16)
    gw, uw = _c(gate_w, np.int8), _c(up_w, np.int8)
    gs, us = _c(gate_s, np.float32), _c(up_s, np.float32)
    offs, tok = _c(row_offsets, np.int32), _c(token_of_row, np.int32)
    T, H = x.shape
    E, I, _ = gw.shape
    M = tok.shape[0]
    if rows is None:
        shape, n, r, c = (M, I), M * I, None, None
    else:
        r, c = _c(rows, np.int64), _c(cols, np.int64)
        shape, n = (r.shape[0],), r.shape[0]
    res = dict(out=np.zeros(shape, np.uint16),
               gate32=np.zeros(shape, np.float32),
               up32=np.zeros(shape, np.float32),
               gabs=np.zeros(shape, np.float64),
               uabs=np.zeros(shape, np.float64))
    rc = _load().q4o_q8_gate_up_swiglu(
        _ptr(x), T, H, I, E, _ptr(gw), _ptr(uw), _ptr(gs), _ptr(us),
        _ptr(offs), _ptr(tok), M, int(silu_mode), n,
        None if r is None else _ptr(r), None if c is None else _ptr(c),
        _ptr(res["out"]), _ptr(res["gate32"]), _ptr(res["up32"]),
        _ptr(res["gabs"]), _ptr(res["uabs"]), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return res


def q8_down_proj(mid_bits, down_w, down_s, row_offsets, rows=None,
                 cols=None, nthreads: int = 0):
    """Q8 down projection (page 52, Q8_DOWN_SOURCE): down_w int8 [E, H, I].
    All M x H outputs or the (rows, cols) elements; a dict with out, out32,
    dabs."""
    mid = _c(mid_bits, np.uint16)
    dw, ds = _c(down_w, np.int8), _c(down_s, np.float32)
    offs = _c(row_offsets, np.int32)
    M, I = mid.shape
    E, H, _ = dw.shape
    if rows is None:
        shape, n, r, c = (M, H), M * H, None, None
    else:
        r, c = _c(rows, np.int64), _c(cols, np.int64)
        shape, n = (r.shape[0],), r.shape[0]
    res = dict(out=np.zeros(shape, np.uint16),
               out32=np.zeros(shape, np.float32),
               dabs=np.zeros(shape, np.float64))
    rc = _load().q4o_q8_down_proj(
        _ptr(mid), M, I, H, E, _ptr(dw), _ptr(ds), _ptr(offs), n,
        None if r is None else _ptr(r), None if c is None else _ptr(c),
        _ptr(res["out"]), _ptr(res["out32"]), _ptr(res["dabs"]),
        int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return res


def trellis_y(state: int) -> int:
    """Code value of one trellis state (page 54, codebook.ts)."""
    return int(_load().q4o_trellis_y(int(state) & 0xFFFFFFFF))


def trellis_scale(scale_f16_bits: int) -> float:
    """The factored row scale RN32(scale * RN32(1/147.800537109375))."""
    return float(_load().q4o_trellis_scale(int(scale_f16_bits)))


def trellis_block(words, Tb: int, k: int, L: int):
    """(states, code values) of the Tb weights of one block of words."""
    w = _c(words, np.uint32)
    st = np.zeros(Tb, np.uint32)
    y = np.zeros(Tb, np.int32)
    lib = _load()
    if (lib.q4o_trellis_block_states(_ptr(w), Tb, k, L, _ptr(st)) != 0 or
            lib.q4o_trellis_block_codes(_ptr(w), Tb, k, L, _ptr(y)) != 0):
        raise ValueError("oracle rejected the block geometry")
    return st, y


def trellis_gate_up_swiglu(x_bits, gate_codes, up_codes, gate_s_f16,
                           up_s_f16, kg: int, ku: int, L: int, Tb: int,
                           row_offsets, token_of_row, rows=None, cols=None,
                           nthreads: int = 0, tail: str = "page"):
    """Trellis gate/up + SwiGLU with factored row scales (page 57,
    gate-up-mma.ts / mixed-gate-up-factored.ts arithmetic).  tail "page":
    the page 52 tail (the pages' equal-width kernels); "mlx": MLX's compiled
    SwiGLU in bf16 arithmetic (the mixed-width kernel).
    gate_codes uint32 [E, I, words], up_codes likewise (widths kg, ku);
    scales f16 bit patterns [E, I].  All M x I outputs or the (rows, cols)
    elements; a dict with out, gate32, up32, gabs, uabs."""
    x = _c(x_bits, np.uint16)
    gc, uc = _c(gate_codes, np.uint32), _c(up_codes, np.uint32)
    gs, us = _c(gate_s_f16, np.uint16), _c(up_s_f16, np.uint16)
    offs, tok = _c(row_offsets, np.int32), _c(token_of_row, np.int32)
    T, H = x.shape
    E, I, _ = gc.shape
    M = tok.shape[0]
    if rows is None:
        shape, n, r, c = (M, I), M * I, None, None
    else:
        r, c = _c(rows, np.int64), _c(cols, np.int64)
        shape, n = (r.shape[0],), r.shape[0]
    res = dict(out=np.zeros(shape, np.uint16),
               gate32=np.zeros(shape, np.float32),
               up32=np.zeros(shape, np.float32),
               gabs=np.zeros(shape, np.float64),
               uabs=np.zeros(shape, np.float64))
    rc = _load().q4o_trellis_gate_up_swiglu(
        _ptr(x), T, H, I, E, _ptr(gc), _ptr(uc), _ptr(gs), _ptr(us),
        int(kg), int(ku), int(L), int(Tb), _ptr(offs), _ptr(tok), M, n,
        None if r is None else _ptr(r), None if c is None else _ptr(c),
        _ptr(res["out"]), _ptr(res["gate32"]), _ptr(res["up32"]),
        _ptr(res["gabs"]), _ptr(res["uabs"]),
        {"page": 0, "mlx": 1}[tail], int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return res
