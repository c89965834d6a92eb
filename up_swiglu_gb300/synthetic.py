"""Seeded synthetic inputs for the fused Q4 MoE gate/up + SwiGLU.

This module only draws numbers: it holds none of the method's arithmetic and
imports nothing else from this package, so the CUDA path and the CPU oracle
can both be fed from it without sharing any code.

Generator: splitmix64 used as a counter-based generator.  Stream ``s`` of
seed ``seed`` is the sequence ``mix(base + (i + 1) * 0x9E3779B97F4A7C15)``,
``i = 0, 1, ...``, where ``base = mix(seed * 0xD1B54A32D192ED03 + s)`` and
``mix`` is the splitmix64 finaliser (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014).

Recipe (the workloads' shapes and value distributions):
- packed Q4 words: uniform 32-bit words, i.e. 8 nibbles uniform in 0..15;
- f32 row scales: ``float32(0.002 + 0.018 * u)``, u uniform in [0, 1);
- activations: Box-Muller normal (f64) times ``x_std``, rounded to f32, then
  to bf16 (round to nearest even on the bit pattern);
- uniform routing: per token, ``topk`` distinct experts drawn uniformly
  without replacement (partial Fisher-Yates);
- Zipf(a) routing: per token, ``topk`` distinct experts drawn one after the
  other with probability proportional to ``rank**-a`` over the experts not
  yet drawn (expert id = rank - 1);
- the exact-integer case: activations integer-valued in [-8, 8], scales
  ``2**-k`` with k uniform in 4..9, so every dot product is exact in f32;
- the down projection's weights and scales follow the same recipe (own
  streams); its exact case draws the intermediate activations as integers
  in [-8, 8] and the scales as ``2**-k``, k uniform in 4..9; measured on
  its own, its input (the intermediate activations) is a Box-Muller normal
  with standard deviation 0.1, rounded to bf16;
- Q8 weights: uniform signed bytes (-128..127, own streams), row scales of
  the Q4 recipe divided by 16 (so that weight times scale spans the same
  range as Q4's nibble - 8 times its scale); the Q8 exact case draws the
  scales as ``2**-k``, k uniform in 8..13;
- trellis codes: uniform 32-bit words (every bit pattern is a valid code
  stream), f16 row scales of the Q4 recipe.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_SEEDMUL = np.uint64(0xD1B54A32D192ED03)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream ids (distinct per array kind)
S_X, S_GATE_W, S_UP_W, S_GATE_S, S_UP_S, S_ROUTE, S_EXACT_X, S_EXACT_S = \
    range(1, 9)
S_DOWN_W, S_DOWN_S, S_EXACT_MID, S_EXACT_DS, S_MID = range(9, 14)
S_Q8_GATE_W, S_Q8_UP_W, S_Q8_DOWN_W = range(14, 17)
S_TR_GATE, S_TR_UP = range(17, 19)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _base(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        b = np.array([seed], dtype=np.uint64) * _SEEDMUL + np.uint64(stream)
        return _mix(b)[0]


def u64(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """Values start .. start+n-1 of stream ``stream`` (uint64)."""
    base = _base(seed, stream)
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix(base + i * _GOLDEN)


def uniform(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """f64 uniform in [0, 1) from the top 53 bits."""
    return (u64(seed, stream, n, start) >> np.uint64(11)).astype(np.float64) \
        * (1.0 / 9007199254740992.0)


def words_u32(seed: int, stream: int, n: int, chunk: int = 1 << 24) -> np.ndarray:
    """n uniform uint32 words (two per 64-bit draw), generated in chunks."""
    out = np.empty(n, dtype=np.uint32)
    n64 = (n + 1) // 2
    for s in range(0, n64, chunk):
        c = min(chunk, n64 - s)
        v = u64(seed, stream, c, start=s).view(np.uint32)
        lo = 2 * s
        hi = min(n, lo + 2 * c)
        out[lo:hi] = v[: hi - lo]
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round f32 to bf16 (nearest, ties to even) and return the bit pattern.
    Input generation only."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        r = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def normal_x(seed: int, T: int, H: int, std: float = 1.0,
             stream: int = S_X) -> np.ndarray:
    """bf16 bits [T, H] of a Box-Muller normal with standard deviation std."""
    n = T * H
    m = (n + 1) // 2
    u1 = 1.0 - uniform(seed, stream, m)            # (0, 1]
    u2 = uniform(seed, stream, m, start=m)
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return f32_to_bf16_bits((z[:n] * std).astype(np.float32)).reshape(T, H)


def weights(seed: int, E: int, I: int, H: int):
    """(gate_w, up_w) uint32 [E, I, H/8] and (gate_s, up_s) f32 [E, I]."""
    assert H % 8 == 0
    n = E * I * (H // 8)
    gate_w = words_u32(seed, S_GATE_W, n).reshape(E, I, H // 8)
    up_w = words_u32(seed, S_UP_W, n).reshape(E, I, H // 8)
    gate_s = (0.002 + 0.018 * uniform(seed, S_GATE_S, E * I)).astype(
        np.float32).reshape(E, I)
    up_s = (0.002 + 0.018 * uniform(seed, S_UP_S, E * I)).astype(
        np.float32).reshape(E, I)
    return gate_w, up_w, gate_s, up_s


def down_weights(seed: int, E: int, H: int, I: int):
    """down_w uint32 [E, H, I/8] and down_s f32 [E, H] (the same recipe as
    gate/up, own streams)."""
    assert I % 8 == 0
    n = E * H * (I // 8)
    down_w = words_u32(seed, S_DOWN_W, n).reshape(E, H, I // 8)
    down_s = (0.002 + 0.018 * uniform(seed, S_DOWN_S, E * H)).astype(
        np.float32).reshape(E, H)
    return down_w, down_s


def exact_down_case(seed: int, M: int, I: int, E: int, H: int):
    """Intermediate activations integer-valued in [-8, 8] (bf16 bits
    [M, I]), power-of-two scales 2**-k, k in 4..9 (f32 [E, H]) and the packed
    words of ``down_weights``: every dot product is an integer below 2**24 in
    magnitude, exact in f32 in any summation order."""
    mi = (u64(seed, S_EXACT_MID, M * I) % np.uint64(17)).astype(np.int64) - 8
    mid = f32_to_bf16_bits(mi.astype(np.float32)).reshape(M, I)
    ks = (u64(seed, S_EXACT_DS, E * H) % np.uint64(6)).astype(np.int64) + 4
    ds = np.ldexp(np.float32(1.0), -ks).astype(np.float32).reshape(E, H)
    down_w, _ = down_weights(seed, E, H, I)
    return mid, down_w, ds


def route_uniform(seed: int, T: int, k: int, E: int) -> np.ndarray:
    """int32 [T, k]: k distinct experts per token, uniform, no replacement."""
    assert 0 < k <= E
    perm = np.tile(np.arange(E, dtype=np.int64), (T, 1))
    u = uniform(seed, S_ROUTE, T * k).reshape(T, k)
    rows = np.arange(T)
    for j in range(k):
        r = j + np.minimum((u[:, j] * (E - j)).astype(np.int64), E - j - 1)
        a = perm[rows, j].copy()
        perm[rows, j] = perm[rows, r]
        perm[rows, r] = a
    return perm[:, :k].astype(np.int32)


def route_zipf(seed: int, T: int, k: int, E: int, a: float) -> np.ndarray:
    """int32 [T, k]: k distinct experts per token, drawn in turn with weight
    rank**-a over the experts not drawn yet (expert id = rank - 1)."""
    assert 0 < k <= E
    w0 = np.arange(1, E + 1, dtype=np.float64) ** (-a)
    u = uniform(seed, S_ROUTE, T * k).reshape(T, k)
    out = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        w = w0.copy()
        for j in range(k):
            c = np.cumsum(w)
            e = int(np.searchsorted(c, u[t, j] * c[-1], side="right"))
            e = min(e, E - 1)
            while w[e] == 0.0:          # guard against an exact cdf edge
                e -= 1
            out[t, j] = e
            w[e] = 0.0
    return out


def exact_integer_case(seed: int, T: int, H: int, E: int, I: int):
    """Activations integer-valued in [-8, 8] (bf16 bits [T, H]) and
    power-of-two scales 2**-k, k in 4..9 (f32 [E, I] each); the packed words
    come from ``weights``.  Every dot product is then an integer below 2**24
    in magnitude, exact in f32 in any summation order."""
    xi = (u64(seed, S_EXACT_X, T * H) % np.uint64(17)).astype(np.int64) - 8
    x = f32_to_bf16_bits(xi.astype(np.float32)).reshape(T, H)
    ks = (u64(seed, S_EXACT_S, 2 * E * I) % np.uint64(6)).astype(np.int64) + 4
    sc = np.ldexp(np.float32(1.0), -ks).astype(np.float32)
    gate_w, up_w, _, _ = weights(seed, E, I, H)
    return x, gate_w, up_w, sc[: E * I].reshape(E, I), sc[E * I:].reshape(E, I)


@dataclass(frozen=True)
class Workload:
    """One synthetic configuration (sizes, routing and value recipe)."""
    name: str
    E: int            # experts
    H: int            # hidden size (K of the projection)
    I: int            # intermediate size (output rows per projection)
    T: int            # tokens
    topk: int         # experts per token
    routing: str      # "single", "uniform" or "zipf"
    zipf_a: float = 0.0
    x_std: float = 1.0
    seed: int = 0
    repeats: int = 1  # independent single-expert calls (decode repeated)

    @property
    def routed_rows(self) -> int:
        return self.T * self.topk


WORKLOADS = {
    # single expert, H=512, I=256, one token (seed 0)
    "expert1_h512_i256_m1": Workload("expert1_h512_i256_m1", 1, 512, 256, 1,
                                     1, "single", seed=0),
    # single expert decode, H=4096, I=1536, one token, the call repeated 1000x
    "expert1_h4096_i1536_m1_x1000": Workload(
        "expert1_h4096_i1536_m1_x1000", 1, 4096, 1536, 1, 1, "single",
        seed=1, repeats=1000),
    # grouped decode: 128 experts, top-8, 32 tokens (256 routed rows)
    "moe128_top8_t32_h5120_i1536": Workload(
        "moe128_top8_t32_h5120_i1536", 128, 5120, 1536, 32, 8, "uniform",
        seed=2),
    # speculative verify: 160 experts, top-8, 8 drafts x 16 sequences
    # (128 tokens, 1024 routed rows), Zipf(1.1) routing
    "moe160_top8_t128_zipf_h5120_i1536": Workload(
        "moe160_top8_t128_zipf_h5120_i1536", 160, 5120, 1536, 128, 8, "zipf",
        zipf_a=1.1, seed=3),
    # prefill: 160 experts, top-8, 4096 tokens (32768 routed rows), x ~ N(0, 0.5^2)
    "moe160_top8_t4096_h5120_i1536": Workload(
        "moe160_top8_t4096_h5120_i1536", 160, 5120, 1536, 4096, 8, "uniform",
        x_std=0.5, seed=4),
}


def routing(w: Workload) -> np.ndarray:
    if w.routing == "single":
        return np.zeros((w.T, w.topk), dtype=np.int32)
    if w.routing == "uniform":
        return route_uniform(w.seed, w.T, w.topk, w.E)
    if w.routing == "zipf":
        return route_zipf(w.seed, w.T, w.topk, w.E, w.zipf_a)
    raise ValueError(w.routing)


def generate(w: Workload, experts: int | None = None, fmt: str = "q4"):
    """x bits [T, H], weights for ``experts`` experts (default w.E; Q4
    words, or Q8 bytes with fmt "q8") and the top-k ids [T, topk]."""
    E = w.E if experts is None else experts
    x = normal_x(w.seed, w.T, w.H, w.x_std)
    gate_w, up_w, gate_s, up_s = (q8_weights if fmt == "q8" else weights)(
        w.seed, E, w.I, w.H)
    return dict(x=x, gate_w=gate_w, up_w=up_w, gate_s=gate_s, up_s=up_s,
                topk=routing(w))


def generate_down(w: Workload, experts: int | None = None, fmt: str = "q4"):
    """The down projection's weights for ``experts`` experts (default w.E)
    and, for measuring it on its own, grouped intermediate activations
    (bf16 bits [routed rows, I], normal with standard deviation 0.1)."""
    E = w.E if experts is None else experts
    down_w, down_s = (q8_down_weights if fmt == "q8" else down_weights)(
        w.seed, E, w.H, w.I)
    mid = normal_x(w.seed, w.routed_rows, w.I, std=0.1, stream=S_MID)
    return dict(down_w=down_w, down_s=down_s, mid=mid)


def _bytes_i8(seed: int, stream: int, n: int) -> np.ndarray:
    return words_u32(seed, stream, (n + 3) // 4).view(np.int8)[:n]


def q8_weights(seed: int, E: int, I: int, H: int):
    """(gate_w, up_w) int8 [E, I, H] and (gate_s, up_s) f32 [E, I]."""
    n = E * I * H
    gate_w = _bytes_i8(seed, S_Q8_GATE_W, n).reshape(E, I, H)
    up_w = _bytes_i8(seed, S_Q8_UP_W, n).reshape(E, I, H)
    gate_s = ((0.002 + 0.018 * uniform(seed, S_GATE_S, E * I)) / 16).astype(
        np.float32).reshape(E, I)
    up_s = ((0.002 + 0.018 * uniform(seed, S_UP_S, E * I)) / 16).astype(
        np.float32).reshape(E, I)
    return gate_w, up_w, gate_s, up_s


def q8_down_weights(seed: int, E: int, H: int, I: int):
    """down_w int8 [E, H, I] and down_s f32 [E, H]."""
    down_w = _bytes_i8(seed, S_Q8_DOWN_W, E * H * I).reshape(E, H, I)
    down_s = ((0.002 + 0.018 * uniform(seed, S_DOWN_S, E * H)) / 16).astype(
        np.float32).reshape(E, H)
    return down_w, down_s


def exact_q8_case(seed: int, T: int, H: int, E: int, I: int):
    """Integer activations in [-8, 8] (bf16 bits [T, H]), the Q8 weights of
    ``q8_weights`` and power-of-two scales 2**-k, k in 8..13: every dot
    product is an integer below 2**24 in magnitude for H <= 16384."""
    xi = (u64(seed, S_EXACT_X, T * H) % np.uint64(17)).astype(np.int64) - 8
    x = f32_to_bf16_bits(xi.astype(np.float32)).reshape(T, H)
    ks = (u64(seed, S_EXACT_S, 2 * E * I) % np.uint64(6)).astype(np.int64) + 8
    sc = np.ldexp(np.float32(1.0), -ks).astype(np.float32)
    gate_w, up_w, _, _ = q8_weights(seed, E, I, H)
    return x, gate_w, up_w, sc[: E * I].reshape(E, I), sc[E * I:].reshape(E, I)


def trellis_weights(seed: int, E: int, I: int, H: int, kg: int, ku: int,
                    block: int = 256):
    """Trellis codes uint32 [E, I, H/block * block*k/32] for gate (kg bits)
    and up (ku bits), and f16 scale bit patterns [E, I] each."""
    gate = words_u32(seed, S_TR_GATE, E * I * (H * kg // 32)).reshape(E, I, -1)
    up = words_u32(seed, S_TR_UP, E * I * (H * ku // 32)).reshape(E, I, -1)
    gs = (0.002 + 0.018 * uniform(seed, S_GATE_S, E * I)).astype(
        np.float16).reshape(E, I).view(np.uint16)
    us = (0.002 + 0.018 * uniform(seed, S_UP_S, E * I)).astype(
        np.float16).reshape(E, I).view(np.uint16)
    return gate, up, gs, us
