"""GPU parity of the down projection and of the whole expert MLP (gate/up,
then down) against the oracle, through the C ABI.

The down projection follows page 52 of "@mlx-bun/inference 0.0.0-stage ->
1.0.0", streamed-experts.ts, DOWN_SOURCE (see tests/parity.py for the
tolerance); exact inputs (integer mid, power-of-two scales) must give
identical bits on every kernel."""
from __future__ import annotations

import numpy as np
import pytest

import harness as hz
import oracle
import parity
from up_swiglu_gb300 import q4moe as q
from up_swiglu_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

KERNELS = [q.KERNEL_AUTO, q.KERNEL_MATVEC, q.KERNEL_GEMM]


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


def _check_down(counts, K, N, kernel=q.KERNEL_AUTO, exact=False, tile=0,
                seed=0, mid_offset=0, **upload_kw):
    p, mid, offs = hz.down_only_problem(seed, counts, K, N, exact=exact)
    d = hz.upload(p, **upload_kw)
    gpu = hz.down(d, offs, mid, kernel=kernel, matvec_tile=tile,
                  mid_offset=mid_offset)
    orc = oracle.down_proj(mid, p.down_w, p.down_s, offs, want_debug=True)
    stats = parity.compare_down(gpu, orc, hz.down_scales(p, offs), K,
                                exact=exact)
    plain = hz.down(d, offs, mid, kernel=kernel, matvec_tile=tile,
                    debug=False)
    assert np.array_equal(plain["out"], gpu["out"])
    return gpu, stats


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("counts,K,N", [([1], 256, 128),
                                        ([3, 0, 8, 1], 512, 256),
                                        ([70, 5, 130], 1536, 384),
                                        ([300], 256, 640)])
def test_down_exact_bit_exact(kernel, counts, K, N):
    """Integer mid and power-of-two scales: identical bits (out and the f32
    value) on the matvec, the GEMM and the automatic mix; N = 384 and 640
    leave the last GEMM tile's second half past the last row."""
    _check_down(counts, K, N, kernel=kernel, exact=True, seed=K + N)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("counts,K,N", [([2, 9, 0, 49, 64], 1536, 512),
                                        ([1, 1, 1], 5120, 256),
                                        ([260, 3], 512, 384)])
def test_down_real_valued(kernel, counts, K, N):
    _, st = _check_down(counts, K, N, kernel=kernel, seed=7 + K)
    assert st["max_err_over_tol"] < 1.0


@pytest.mark.parametrize("tile", [16, 32, 64, 128])
def test_down_matvec_tiles(tile):
    """Every unit height: bit-identical on exact inputs, within the bound on
    real ones; N = 272 (17 blocks of 16) leaves ragged tiles at every
    height, including a second half wholly past the last row."""
    ref, _ = _check_down([5, 8, 0, 3], 512, 272, kernel=q.KERNEL_MATVEC,
                         exact=True, seed=3)
    got, _ = _check_down([5, 8, 0, 3], 512, 272, kernel=q.KERNEL_MATVEC,
                         exact=True, tile=tile, seed=3)
    assert np.array_equal(got["out"], ref["out"])
    _check_down([5, 8, 0, 3], 512, 272, kernel=q.KERNEL_MATVEC, tile=tile,
                seed=4)


@pytest.mark.parametrize("K,N", [(200, 40), (264, 64), (384, 24)])
def test_down_generic_shapes(K, N):
    """K % 256 != 0 or N % 16 != 0: the generic down kernel (the GEMM needs
    K % 64 == 0 and N % 128 == 0 and is refused here)."""
    _check_down([2, 7, 1], K, N, kernel=q.KERNEL_MATVEC, exact=True, seed=K)
    _check_down([2, 7, 1], K, N, seed=K + 1)
    p, mid, offs = hz.down_only_problem(1, [2, 7, 1], K, N)
    d = hz.upload(p)
    with pytest.raises(q.Q4moeError) as ei:
        hz.down(d, offs, mid, kernel=q.KERNEL_GEMM)
    assert ei.value.code == q.ERR_INVALID_ARG


@pytest.mark.parametrize("kernel", [q.KERNEL_MATVEC, q.KERNEL_GEMM])
def test_down_pointer_table_and_unaligned_mid(kernel):
    """Slabs through a per-expert pointer table (shuffled slots), and mid
    16 bytes past a 256-byte boundary."""
    _check_down([4, 0, 66, 9], 512, 256, kernel=kernel, exact=True, seed=11,
                ptr_table=True, mid_offset=8)
    _check_down([4, 0, 66, 9], 512, 256, kernel=kernel, seed=12,
                ptr_table=True, mid_offset=8)


def test_down_empty_and_single_row():
    import torch
    p, mid, offs = hz.down_only_problem(2, [1], 1536, 5120)
    d = hz.upload(p)
    gpu = hz.down(d, offs, mid)
    orc = oracle.down_proj(mid, p.down_w, p.down_s, offs, want_debug=True)
    parity.compare_down(gpu, orc, hz.down_scales(p, offs), 1536)
    # M = 0 is a no-op
    out = torch.full((1, 5120), 7, dtype=torch.int16, device="cuda")
    q.q4moe_down_proj(None, d.slabs, torch.zeros(2, dtype=torch.int32,
                                                 device="cuda"),
                      0, 5120, 1536, out)
    torch.cuda.synchronize()
    assert torch.all(out == 7)


@pytest.mark.parametrize("kernel", KERNELS)
def test_down_bad_offsets_raise_status(kernel):
    import torch
    p, mid, offs = hz.down_only_problem(5, [3, 70], 256, 256)
    d = hz.upload(p)
    bad = offs.copy()
    bad[1] = 80                           # decreasing, past M
    gpu = hz.down(d, bad, mid, kernel=kernel, debug=False)
    assert q.q4moe_device_status(clear=True) & q.DEV_BAD_ROW_OFFSETS
    assert np.all(gpu["out"] == 0xFFFF)   # nothing written
    torch.cuda.synchronize()


@pytest.mark.parametrize("counts,K,N,exact", [([1], 1536, 4096, False),
                                              ([5], 1536, 4096, True),
                                              ([8], 512, 4864, True),
                                              ([3], 256, 4600, True),
                                              ([2], 5120, 1024, False)])
def test_down_single_expert_latency_kernel(counts, K, N, exact):
    """One expert with at most 8 rows (the single-sequence decode): the
    kernel laid out for latency (each CTA a few output rows, K split over
    its warps).  N = 4864 gives every CTA 32 rows (two m16 tiles), N = 4600
    a last CTA of 12 rows; the matvec choice runs the same kernel."""
    _check_down(counts, K, N, exact=exact, seed=K + N)
    _check_down(counts, K, N, kernel=q.KERNEL_MATVEC, exact=exact,
                seed=K + N)


def test_down_single_expert_bad_offsets():
    """The latency kernel checks the one expert's offsets {0, M}: a wrong
    pair raises the status bit and nothing is written."""
    p, mid, offs = hz.down_only_problem(9, [4], 512, 1024)
    d = hz.upload(p)
    bad = offs.copy()
    bad[1] = 3
    gpu = hz.down(d, bad, mid, debug=False)
    assert q.q4moe_device_status(clear=True) & q.DEV_BAD_ROW_OFFSETS
    assert np.all(gpu["out"] == 0xFFFF)


# ------------------------------------------------------------ expert MLP --

def _mlp_problem(seed, E, I, H, T, k, exact):
    p = hz.exact_problem(seed, E, I, H, T, k) if exact else \
        hz.random_problem(seed, E, I, H, T, k)
    return hz.with_down(p, seed, exact=exact)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("E,I,H,T,k", [(1, 256, 512, 1, 1),
                                       (6, 512, 256, 40, 3),
                                       (3, 256, 512, 200, 2)])
def test_mlp_exact_mid_then_down(kernel, E, I, H, T, k):
    """Exact gate/up inputs: mid is bit-identical to the oracle's; the down
    outputs then meet the down bound against the oracle's down of the
    oracle's mid."""
    p = _mlp_problem(E + I, E, I, H, T, k, exact=True)
    d = hz.upload(p)
    offs_d, tok_d, _ = hz.group(d)
    offs, tok = offs_d.cpu().numpy(), tok_d.cpu().numpy()
    gpu = hz.expert_mlp(d, offs_d, tok_d, kernel=kernel)
    orc_mid = oracle.gate_up_swiglu(p.x, p.gate_w, p.up_w, p.gate_s, p.up_s,
                                    offs, tok)
    assert np.array_equal(gpu["mid"], orc_mid)
    orc = oracle.down_proj(orc_mid, p.down_w, p.down_s, offs,
                           want_debug=True)
    parity.compare_down_bits(gpu["out"], orc, hz.down_scales(p, offs), I)
    # the two calls in turn give the same bits as the fused one
    sep = hz.down(d, offs_d, hz.gate_up(d, offs_d, tok_d, kernel=kernel,
                                        debug=False)["out"], kernel=kernel,
                  debug=False)
    assert np.array_equal(sep["out"], gpu["out"])


@pytest.mark.parametrize("kernel", KERNELS)
def test_mlp_real_valued(kernel):
    """Real inputs: mid meets the gate/up bound; each down output lies
    within the down bound plus the effect of every mid rounding the oracle
    shows could go either way (computed from the oracle alone)."""
    E, I, H, T, k = 5, 512, 768, 48, 4
    p = _mlp_problem(31, E, I, H, T, k, exact=False)
    d = hz.upload(p)
    offs_d, tok_d, _ = hz.group(d)
    offs, tok = offs_d.cpu().numpy(), tok_d.cpu().numpy()
    gpu = hz.expert_mlp(d, offs_d, tok_d, kernel=kernel, workspace=True)
    og = oracle.gate_up_swiglu(p.x, p.gate_w, p.up_w, p.gate_s, p.up_s,
                               offs, tok, want_debug=True)
    gs, us = hz.element_scales(p, offs)
    parity.compare({"out": gpu["mid"], "gate32": gpu["gate32"],
                    "up32": gpu["up32"]}, og, gs, us, H)
    allow = parity.mid_flip_allowance(og, gs, us, H)          # [M, I]
    orc = oracle.down_proj(og["out"], p.down_w, p.down_s, offs,
                           want_debug=True)
    k_ = np.arange(I)
    W = np.abs(((p.down_w[:, :, k_ // 8] >> (4 * (k_ % 8)).astype(np.uint32))
                & 0xF).astype(np.float64) - 8.0)               # [E, H, I]
    eo = np.repeat(np.arange(E), np.diff(offs))
    extra = np.stack([W[eo[r]] @ allow[r] for r in range(len(eo))]) * \
        hz.down_scales(p, offs)
    parity.compare_down_bits(gpu["out"], orc, hz.down_scales(p, offs), I,
                             extra_tol=extra)


@pytest.mark.parametrize("name", ["moe128_top8_t32_h5120_i1536",
                                  "moe160_top8_t4096_h5120_i1536"])
def test_mlp_full_size_sampled(name):
    """The full decode and prefill configurations: the fused MLP's mid and
    out on sampled rows, every column of each, against the oracle (mid rows
    computed one by one, then their down outputs)."""
    w = syn.WORKLOADS[name]
    g = syn.generate(w)
    p = hz.with_down(hz.Problem(g["x"], g["gate_w"], g["up_w"], g["gate_s"],
                                g["up_s"], g["topk"]), w.seed)
    d = hz.upload(p)
    offs_d, tok_d, _ = hz.group(d)
    offs, tok = offs_d.cpu().numpy(), tok_d.cpu().numpy()
    gpu = hz.expert_mlp(d, offs_d, tok_d, workspace=True)
    M = gpu["out"].shape[0]
    assert M == w.routed_rows
    assert np.all(((gpu["out"] >> 7) & 0xFF) != 0xFF)
    rng = np.random.default_rng(M)
    rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, 6)]))
    rr = np.repeat(rows, w.I)
    cc = np.tile(np.arange(w.I), rows.size)
    og = oracle.gate_up_swiglu_sampled(p.x, p.gate_w, p.up_w, p.gate_s,
                                       p.up_s, offs, tok, rr, cc)
    gs, us = hz.element_scales(p, offs)
    parity.compare({"out": gpu["mid"][rr, cc], "gate32": gpu["gate32"][rr, cc],
                    "up32": gpu["up32"][rr, cc]}, og,
                   gs[rr, cc], us[rr, cc], w.H)
    # the down outputs of those rows, from the oracle's mid rows
    mid_o = np.zeros((M, w.I), np.uint16)
    mid_o[rr, cc] = og["out"]
    allow = np.zeros((M, w.I))
    allow[rr, cc] = parity.mid_flip_allowance(
        og, gs[rr, cc], us[rr, cc], w.H)
    hr = np.repeat(rows, w.H)
    hc = np.tile(np.arange(w.H), rows.size)
    orc = oracle.down_proj_sampled(mid_o, p.down_w, p.down_s, offs, hr, hc)
    k_ = np.arange(w.I)
    eo = np.repeat(np.arange(p.E), np.diff(offs))
    extra = np.zeros(hr.size)
    for j, r in enumerate(rows):
        Wr = np.abs(((p.down_w[eo[r]][:, k_ // 8] >>
                      (4 * (k_ % 8)).astype(np.uint32)) & 0xF)
                    .astype(np.float64) - 8.0)
        extra[j * w.H:(j + 1) * w.H] = (Wr @ allow[r]) * p.down_s[eo[r]]
    ds = hz.down_scales(p, offs)
    parity.compare_down_bits(gpu["out"][hr, hc], orc, ds[hr, hc], w.I,
                             extra_tol=extra)
