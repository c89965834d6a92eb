"""GPU parity of the trellis (QTIP 1MAD) gate/up + SwiGLU against the
oracle, through the C ABI (q4moe_trellis_gate_up_swiglu).

Pages of "@mlx-bun/inference 0.0.0-stage -> 1.0.0": page 57, trellis/
gate-up-mma.ts and mixed-gate-up-factored.ts (factored row scale; the
mixed-width kernel ends with MLX's compiled SwiGLU, the default tail when
gate and up widths differ), page 54, trellis/codebook.ts (state and code
value).  Integer activations in [-2, 2] make every sum exact, so those
cases must give the oracle's bits; real inputs meet the bound of
tests/parity.py."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import parity
import harness as hz
from up_swiglu_gb300 import q4moe as q
from up_swiglu_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

TB = 256


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    q.load()
    oracle.build()
    q.q4moe_device_status(clear=True)
    yield
    assert q.q4moe_device_status(clear=True) == 0, "device status raised"


def _problem(seed, counts, I, H, kg, ku, exact=False):
    """One token per grouped row, expert e getting counts[e] rows (a row's
    codes are H * k / 32 words whatever the block size)."""
    E, M = len(counts), int(sum(counts))
    rng = np.random.default_rng(seed)
    gc = syn.words_u32(seed, 40, E * I * (H * kg // 32)).reshape(E, I, -1)
    uc = syn.words_u32(seed, 41, E * I * (H * ku // 32)).reshape(E, I, -1)
    gs = (0.002 + 0.018 * rng.random((E, I))).astype(np.float16)
    us = (0.002 + 0.018 * rng.random((E, I))).astype(np.float16)
    if exact:
        x = syn.f32_to_bf16_bits(
            rng.integers(-2, 3, size=(max(M, 1), H)).astype(np.float32))
    else:
        x = syn.normal_x(seed, max(M, 1), H)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    tok = rng.permutation(max(M, 1))[:M].astype(np.int32)
    return dict(x=x, gc=gc, uc=uc, gs=gs.view(np.uint16),
                us=us.view(np.uint16), offs=offs, tok=tok, I=I, H=H, kg=kg,
                ku=ku)


def _auto_tail(p):
    """The tail Q4MOE_TAIL_AUTO takes: the pages' mixed-width kernel's
    (MLX) when the widths differ, page 52's otherwise."""
    return "mlx" if p["kg"] != p["ku"] else "page"


def _run(p, L=12, ptr_table=False, debug=True, tb=TB, tail=None):
    import torch
    E = p["gc"].shape[0]
    lay = q.q4moe_trellis_canonical_layout(p["H"], p["I"], tb, L, p["kg"],
                                           p["ku"])
    host = q.pack_trellis_pool(lay, p["gc"], p["uc"], p["gs"], p["us"])
    buf, pool = hz.aligned_device_buffer(host.size)
    pool.copy_(torch.from_numpy(host.reshape(-1)))
    keep = [buf]
    if ptr_table:
        perm = np.random.default_rng(E).permutation(E)
        buf2, pool2 = hz.aligned_device_buffer(host.size)
        keep.append(buf2)
        for e in range(E):
            n = lay.slab_bytes
            pool2[perm[e] * n:(perm[e] + 1) * n].copy_(
                pool[e * n:(e + 1) * n])
        ptrs = torch.tensor([pool2.data_ptr() + int(perm[e]) * lay.slab_bytes
                             for e in range(E)], dtype=torch.int64,
                            device="cuda")
        keep.append(ptrs)
        slabs = q.make_trellis_slabs(E, lay, slab_ptrs=ptrs)
    else:
        slabs = q.make_trellis_slabs(E, lay, base=pool)
    M, I, H = len(p["tok"]), p["I"], p["H"]
    xd = torch.from_numpy(p["x"].view(np.int16)).cuda()
    out = torch.full((max(M, 1), I), -1, dtype=torch.int16, device="cuda")
    o = q.q4moe_options_t()
    o.num_tokens = p["x"].shape[0]
    if tail is not None:
        o.tail = {"page": q.TAIL_PAGE, "mlx": q.TAIL_MLX}[tail]
    g32 = torch.full((max(M, 1), I), float("nan"), device="cuda")
    u32 = torch.full((max(M, 1), I), float("nan"), device="cuda")
    if debug:
        o.gate_f32, o.up_f32 = g32.data_ptr(), u32.data_ptr()
    q.q4moe_trellis_gate_up_swiglu(xd, slabs, torch.from_numpy(p["offs"])
                                   .cuda(), torch.from_numpy(p["tok"]).cuda(),
                                   M, H, I, out, o)
    torch.cuda.synchronize()
    res = {"out": out[:M].cpu().numpy().view(np.uint16)}
    if debug:
        res["gate32"] = g32[:M].cpu().numpy()
        res["up32"] = u32[:M].cpu().numpy()
    return res


def _compare(p, gpu, L=12, exact=False, tb=TB, tail=None):
    tail = tail or _auto_tail(p)
    orc = oracle.trellis_gate_up_swiglu(p["x"], p["gc"], p["uc"], p["gs"],
                                        p["us"], p["kg"], p["ku"], L, tb,
                                        p["offs"], p["tok"], tail=tail)
    e_of = np.repeat(np.arange(len(p["offs"]) - 1), np.diff(p["offs"]))
    rcp = np.float32(1.0 / 147.800537109375)
    fs = lambda s: (s.view(np.float16).astype(np.float32) * rcp  # noqa: E731
                    ).astype(np.float32)
    gsc, usc = fs(p["gs"])[e_of], fs(p["us"])[e_of]
    return parity.compare(gpu, orc, gsc, usc, p["H"], exact=exact,
                          tail=tail)


@pytest.mark.parametrize("kg,ku", [(4, 4), (2, 4), (3, 2), (3, 3), (2, 2),
                                   (1, 6)])
def test_trellis_exact_bit_exact(kg, ku):
    """Templated widths (2, 3, 4 in any pair) and the general kernel
    (1 and 6 bits)."""
    p = _problem(kg * 10 + ku, [3, 0, 9, 1, 20], 64, 512, kg, ku, exact=True)
    gpu = _run(p)
    _compare(p, gpu, exact=True)
    assert np.array_equal(_run(p, debug=False)["out"], gpu["out"])


@pytest.mark.parametrize("kg,ku,L", [(4, 4, 12), (2, 3, 12), (4, 2, 16),
                                     (3, 3, 8)])
def test_trellis_real_valued(kg, ku, L):
    p = _problem(100 + kg + ku + L, [1, 7, 2, 13], 96, 1024, kg, ku)
    _compare(p, _run(p, L=L), L=L)


@pytest.mark.parametrize("tb,kg,ku,L", [(32, 4, 4, 12), (128, 2, 3, 12),
                                        (64, 2, 2, 24), (512, 3, 4, 12)])
def test_trellis_block_sizes_and_windows(tb, kg, ku, L):
    """Blocks of 32 (one run a block), 128, 64 with a 24-bit window over
    2-bit codes (the window spans more than one block's worth of words of
    a run), and 512."""
    p = _problem(tb + L, [4, 9, 0, 2], 48, 1024, kg, ku, exact=True)
    _compare(p, _run(p, L=L, tb=tb), L=L, exact=True, tb=tb)
    p = _problem(tb + L + 1, [4, 9, 0, 2], 48, 1024, kg, ku)
    _compare(p, _run(p, L=L, tb=tb), L=L, tb=tb)


def test_trellis_pointer_table_and_bad_offsets():
    import torch
    p = _problem(7, [2, 5, 0, 3], 32, 256, 4, 4, exact=True)
    _compare(p, _run(p, ptr_table=True), exact=True)
    bad = dict(p)
    bad["offs"] = np.array([0, 6, 2, 7, 10], np.int32)    # decreasing
    out = _run(bad, debug=False)["out"]
    assert q.q4moe_device_status(clear=True) & q.DEV_BAD_ROW_OFFSETS
    assert np.all(out == 0xFFFF)
    torch.cuda.synchronize()


def test_trellis_full_size_decode_sampled():
    """The grouped-decode size (128 experts, top-8, 32 tokens, H = 5120,
    I = 1536) with 4-bit gate and 3-bit up codes: sampled outputs and whole
    rows against the oracle."""
    w = syn.WORKLOADS["moe128_top8_t32_h5120_i1536"]
    topk = syn.route_uniform(w.seed, w.T, w.topk, w.E)
    offs, tok, _ = oracle.group_rows(topk, w.E)
    counts = np.diff(offs)
    p = _problem(w.seed, counts, w.I, w.H, 4, 3)
    p["x"] = syn.normal_x(w.seed, w.T, w.H)
    p["tok"] = tok
    gpu = _run(p)
    M, I = gpu["out"].shape
    rng = np.random.default_rng(M)
    rows = np.concatenate([rng.integers(0, M, 1500), np.zeros(I, int),
                           np.full(I, M - 1)])
    cols = np.concatenate([rng.integers(0, I, 1500), np.arange(I),
                           np.arange(I)])
    orc = oracle.trellis_gate_up_swiglu(p["x"], p["gc"], p["uc"], p["gs"],
                                        p["us"], 4, 3, 12, TB, offs, tok,
                                        rows, cols, tail="mlx")
    e_of = np.repeat(np.arange(w.E), counts)
    rcp = np.float32(1.0 / 147.800537109375)
    gsc = (p["gs"].view(np.float16).astype(np.float32) * rcp)[e_of]
    usc = (p["us"].view(np.float16).astype(np.float32) * rcp)[e_of]
    sel = {k: gpu[k][rows, cols] for k in ("out", "gate32", "up32")}
    parity.compare(sel, orc, gsc[rows, cols], usc[rows, cols], w.H,
                   tail="mlx")


# ------------------------------------------------------------ MLX tail --

def test_mlx_tail_exhaustive_bf16():
    """All finite bf16 gate values, several up values: the device's MLX
    tail (its sigmoid table) equals the oracle's bit for bit."""
    import torch
    g = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    g = g[((g >> 7) & 0xFF) != 0xFF]
    for up in (1.0, -3.0, 0.0078125, 250.0):
        u = np.full(g.shape, syn.f32_to_bf16_bits(np.float32([up]))[0],
                    np.uint16)
        gd = torch.from_numpy(g.view(np.int16)).cuda()
        ud = torch.from_numpy(u.view(np.int16)).cuda()
        res = torch.empty((g.size, 4), dtype=torch.int16, device="cuda")
        q.q4moe_debug_tail_mlx(gd, ud, g.size, res)
        r = res.cpu().numpy().view(np.uint16)
        t = oracle.tail_mlx_array(syn.bf16_bits_to_f32(g),
                                  syn.bf16_bits_to_f32(u))
        assert np.array_equal(r[:, 3], r[:, 0])
        for col, name in ((0, "sigmoid"), (1, "silu"), (2, "out")):
            bad = np.flatnonzero(r[:, col] != t[:, col + 2])
            assert bad.size == 0, f"{name}: {bad.size} differ, e.g. gate " \
                f"{g[bad[:4]]}"


@pytest.mark.parametrize("kg,ku,tail", [(4, 4, "mlx"), (3, 3, "mlx"),
                                        (2, 4, "page"), (4, 3, "page"),
                                        (4, 3, "mlx"), (2, 2, "page")])
def test_trellis_tail_choice(kg, ku, tail):
    """The tail asked for in the options, whatever the widths (AUTO's choice
    is covered by every other test): bit-exact on exact inputs, within the
    bound on real ones."""
    p = _problem(kg * 10 + ku + 7, [3, 0, 9, 1, 20], 64, 512, kg, ku,
                 exact=True)
    _compare(p, _run(p, tail=tail), exact=True, tail=tail)
    p = _problem(kg * 10 + ku + 8, [1, 7, 2, 13], 96, 1024, kg, ku)
    _compare(p, _run(p, tail=tail), tail=tail)


def test_mlx_and_page_tails_differ_on_device():
    """The choice is live: with gate values spread over the sigmoid's curve,
    the two tails give different outputs somewhere."""
    p = _problem(91, [8, 8], 64, 512, 4, 3)
    a = _run(p, tail="page", debug=False)["out"]
    b = _run(p, tail="mlx", debug=False)["out"]
    assert np.any(a != b)
