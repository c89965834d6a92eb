"""GPU parity of the Q8 weight format (signed bytes) against the oracle.

Page 52 of "@mlx-bun/inference 0.0.0-stage -> 1.0.0", streamed-experts.ts,
Q8_GATE_UP_SOURCE and Q8_DOWN_SOURCE: the same contract as Q4 with one
signed byte per weight and no zero point.  Exact inputs (integer
activations, power-of-two scales) must give the oracle's bits on every
kernel; real-valued inputs meet the bound of tests/parity.py."""
from __future__ import annotations

import numpy as np
import pytest

import harness as hz
import oracle
import parity
from up_swiglu_gb300 import q4moe as q
from up_swiglu_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

KERNELS = [q.KERNEL_AUTO, q.KERNEL_MATVEC, q.KERNEL_GEMM,
           q.KERNEL_BATCH_INVARIANT]


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


def _scale_bf16(x, shift):
    f = syn.bf16_bits_to_f32(x).astype(np.float64) * 2.0 ** shift
    return syn.f32_to_bf16_bits(f.astype(np.float32))


def _check(p, kernel=q.KERNEL_AUTO, exact=False, tile=0, workspace=False,
           **upload_kw):
    d = hz.upload(p, layout=hz.q8_layout(p), **upload_kw)
    offs_d, tok_d, _ = hz.group(d)
    offs, tok = offs_d.cpu().numpy(), tok_d.cpu().numpy()
    gpu = hz.gate_up(d, offs_d, tok_d, kernel=kernel, matvec_tile=tile,
                     workspace=workspace)
    orc = oracle.q8_gate_up_swiglu(p.x, p.gate_w, p.up_w, p.gate_s, p.up_s,
                                   offs, tok)
    gs, us = hz.element_scales(p, offs)
    stats = parity.compare(gpu, orc, gs, us, p.H, exact=exact)
    plain = hz.gate_up(d, offs_d, tok_d, kernel=kernel, matvec_tile=tile,
                       debug=False)
    assert np.array_equal(plain["out"], gpu["out"])
    return gpu, stats


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("E,I,H,T,k", [(1, 256, 512, 1, 1),
                                       (4, 512, 1024, 40, 2),
                                       (3, 256, 512, 200, 2),
                                       (2, 128, 5120, 3, 1)])
def test_q8_gate_up_exact_bit_exact(kernel, E, I, H, T, k):
    p = hz.q8_problem(E + H, E, I, H, T, k, exact=True)
    _check(p, kernel=kernel, exact=True)


@pytest.mark.parametrize("kernel", KERNELS)
def test_q8_gate_up_real_valued(kernel):
    p = hz.q8_problem(31, 6, 512, 2048, 64, 4)
    _check(p, kernel=kernel)
    _check(p, kernel=kernel, workspace=True)


@pytest.mark.parametrize("tile", [16, 32, 64, 128])
def test_q8_matvec_tiles(tile):
    p = hz.q8_counts_problem(5, [5, 8, 0, 3, 9], 272, 1024, exact=True)
    ref, _ = _check(p, kernel=q.KERNEL_MATVEC, exact=True)
    got, _ = _check(p, kernel=q.KERNEL_MATVEC, exact=True, tile=tile)
    assert np.array_equal(got["out"], ref["out"])
    p = hz.q8_counts_problem(6, [5, 8, 0, 3, 9], 272, 1024)
    _check(p, kernel=q.KERNEL_MATVEC, tile=tile)


@pytest.mark.parametrize("shift", [40, -60, -90])
def test_q8_matvec_scaled_exact_activations(shift):
    """f16 staging under a power-of-two scale (40, -60) and the bf16 path
    (-90); every sum exact, so the oracle's bits."""
    p = hz.q8_counts_problem(7, [5, 8, 1, 3], 128, 512, exact=True)
    p.x = _scale_bf16(p.x, shift)
    _check(p, kernel=q.KERNEL_MATVEC, exact=True)


def test_q8_matvec_wide_span_and_subnormal_fall_back_to_bf16():
    p = hz.q8_counts_problem(8, [2, 3], 128, 512, exact=True)
    rows = np.flatnonzero(p.topk[:, 0] == 0)
    p.x[rows[0]] = _scale_bf16(p.x[rows[0]][None], 20)[0]
    p.x[rows[1]] = _scale_bf16(p.x[rows[1]][None], -20)[0]
    _check(p, kernel=q.KERNEL_MATVEC, exact=True)
    p = hz.q8_counts_problem(9, [3, 2], 256, 1024)
    p.x[0, 5] = 0x0001
    p.x[1, 7] = 0x8003
    _check(p, kernel=q.KERNEL_MATVEC)


@pytest.mark.parametrize("H,I", [(196, 20), (388, 64), (1152, 36)])
def test_q8_generic_shapes(H, I):
    """H % 128 != 0 or I % 16 != 0: the generic kernel (the GEMM, needing
    H % 64 == 0 and I % 128 == 0, is refused for these shapes)."""
    p = hz.q8_counts_problem(H, [2, 7, 1], I, H, exact=True)
    _check(p, kernel=q.KERNEL_MATVEC, exact=True)
    p = hz.q8_counts_problem(H + 1, [2, 7, 1], I, H)
    _check(p)


@pytest.mark.parametrize("kernel", [q.KERNEL_MATVEC, q.KERNEL_GEMM])
def test_q8_pointer_table(kernel):
    p = hz.q8_counts_problem(10, [4, 0, 70, 9], 256, 512, exact=True)
    _check(p, kernel=kernel, exact=True, ptr_table=True)


# ------------------------------------------------------------ down, MLP --

def _check_down(counts, K, N, kernel=q.KERNEL_AUTO, exact=False, tile=0,
                seed=0):
    p, mid, offs = hz.q8_down_only_problem(seed, counts, K, N, exact=exact)
    d = hz.upload(p, layout=hz.q8_layout(p))
    gpu = hz.down(d, offs, mid, kernel=kernel, matvec_tile=tile)
    orc = oracle.q8_down_proj(mid, p.down_w, p.down_s, offs)
    parity.compare_down(gpu, orc, hz.down_scales(p, offs), K, exact=exact)
    return gpu


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("counts,K,N", [([1], 256, 128), ([3, 0, 70, 1], 512, 384),
                                        ([9, 2], 1536, 272), ([5], 1536, 4600)])
def test_q8_down(kernel, counts, K, N):
    if kernel == q.KERNEL_GEMM and N % 128:
        pytest.skip("the GEMM needs N % 128 == 0")
    _check_down(counts, K, N, kernel=kernel, exact=True, seed=K + N)
    _check_down(counts, K, N, kernel=kernel, seed=K + N + 1)


@pytest.mark.parametrize("kernel", KERNELS)
def test_q8_mlp_exact_mid_then_down(kernel):
    p = hz.q8_problem(44, 4, 256, 512, 60, 2, exact=True)
    d = hz.upload(p, layout=hz.q8_layout(p))
    offs_d, tok_d, _ = hz.group(d)
    offs, tok = offs_d.cpu().numpy(), tok_d.cpu().numpy()
    gpu = hz.expert_mlp(d, offs_d, tok_d, kernel=kernel)
    orc_mid = oracle.q8_gate_up_swiglu(p.x, p.gate_w, p.up_w, p.gate_s,
                                       p.up_s, offs, tok)["out"]
    assert np.array_equal(gpu["mid"], orc_mid)
    orc = oracle.q8_down_proj(orc_mid, p.down_w, p.down_s, offs)
    parity.compare_down_bits(gpu["out"], orc, hz.down_scales(p, offs), p.I)


@pytest.mark.parametrize("M", [1, 4, 8])
def test_q8_single_expert_latency_kernel(M):
    """Q8, one expert with 1 to 8 rows (the kernel laid out for latency):
    K = 160 (rows of 160 bytes), I = 100 (one row per CTA); exact and
    real-valued against the Q8 oracle."""
    for exact in (True, False):
        p = hz.q8_counts_problem(50 + M, [M], 100, 160, exact=exact)
        _check(p, exact=exact)


def test_q8_full_size_decode_sampled():
    """Q8 at the grouped-decode size (128 experts, top-8, 32 tokens,
    H = 5120, I = 1536): sampled outputs and whole rows against the
    oracle."""
    w = syn.WORKLOADS["moe128_top8_t32_h5120_i1536"]
    p = hz.q8_problem(w.seed, w.E, w.I, w.H, w.T, w.topk, with_down=False)
    d = hz.upload(p, layout=hz.q8_layout(p))
    offs_d, tok_d, _ = hz.group(d)
    offs, tok = offs_d.cpu().numpy(), tok_d.cpu().numpy()
    gpu = hz.gate_up(d, offs_d, tok_d, workspace=True)
    M, I = gpu["out"].shape
    rng = np.random.default_rng(M)
    rows = np.concatenate([rng.integers(0, M, 2000), np.zeros(I, int),
                           np.full(I, M - 1)])
    cols = np.concatenate([rng.integers(0, I, 2000), np.arange(I),
                           np.arange(I)])
    orc = oracle.q8_gate_up_swiglu(p.x, p.gate_w, p.up_w, p.gate_s, p.up_s,
                                   offs, tok, rows, cols)
    gs, us = hz.element_scales(p, offs)
    sel = {k: gpu[k][rows, cols] for k in ("out", "gate32", "up32")}
    parity.compare(sel, orc, gs[rows, cols], us[rows, cols], p.H)
