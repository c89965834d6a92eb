"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every test here runs libq4moe's kernels on cuda:0 and compares with the
oracle on the same seeded inputs (see tests/parity.py for the tolerance)."""
from __future__ import annotations

import numpy as np
import pytest

import harness as hz
import oracle
import parity
from up_swiglu_gb300 import q4moe as q
from up_swiglu_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    q.load()                 # builds if missing; raises if it cannot load
    oracle.build()
    q.q4moe_device_status(clear=True)
    yield
    assert q.q4moe_device_status(clear=True) == 0, "device status raised"


def _oracle_full(p, offs, tok):
    return oracle.gate_up_swiglu(p.x, p.gate_w, p.up_w, p.gate_s, p.up_s,
                                 offs, tok, want_debug=True)


def _run_and_compare(p, kernel=q.KERNEL_AUTO, exact=False, matvec_tile=0,
                     **upload_kw):
    d = hz.upload(p, **upload_kw)
    offs_d, tok_d, _ = hz.group(d)
    offs, tok = offs_d.cpu().numpy(), tok_d.cpu().numpy()
    o_offs, o_tok, _ = oracle.group_rows(p.topk, p.E)
    assert np.array_equal(offs, o_offs) and np.array_equal(tok, o_tok)
    gpu = hz.gate_up(d, offs_d, tok_d, kernel=kernel, matvec_tile=matvec_tile)
    orc = _oracle_full(p, offs, tok)
    gs, us = hz.element_scales(p, offs)
    stats = parity.compare(gpu, orc, gs, us, p.H, exact=exact)
    # the plain entry point (no debug outputs) writes the same bits
    plain = hz.gate_up(d, offs_d, tok_d, kernel=kernel, debug=False,
                       matvec_tile=matvec_tile)
    assert np.array_equal(plain["out"], gpu["out"])
    # the matvec's unit height only changes the f32 summation order: every
    # height meets the same bound (and exact sums give the same bits)
    if not matvec_tile and kernel != q.KERNEL_GEMM:
        for tile in (16, 128):
            tiled = hz.gate_up(d, offs_d, tok_d, kernel=kernel,
                               matvec_tile=tile)
            parity.compare(tiled, orc, gs, us, p.H, exact=exact)
            if exact:
                assert np.array_equal(tiled["out"], gpu["out"])
    # with a workspace the GEMM reads the grouped rows through TMA: same bits
    ws = hz.gate_up(d, offs_d, tok_d, kernel=kernel, workspace=True,
                    matvec_tile=matvec_tile)
    assert np.array_equal(ws["out"], gpu["out"])
    assert np.array_equal(ws["gate32"].view(np.uint32),
                          gpu["gate32"].view(np.uint32))
    return stats


# ----------------------------------------------------------------- grouping --

@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (0, 8, 4), (5, 3, 7),
                                   (1000, 8, 160), (4096, 8, 160),
                                   (300, 2, 1024), (2047, 1, 3),
                                   (4096, 4, 1024), (20000, 8, 7)])
def test_group_rows_matches_oracle(T, k, E):
    """Small inputs take one thread block; large ones (here 32768, 16384
    and 160000 pairs) are counted, scanned and scattered by many blocks."""
    import torch
    rng = np.random.default_rng(T + E)
    topk = rng.integers(0, E, size=(T, k)).astype(np.int32)
    p = hz.Problem(np.zeros((T, 8), np.uint16), np.zeros((E, 4, 1), np.uint32),
                   None, None, None, topk)
    d = hz.DeviceProblem(p, None, None)
    d.topk = torch.from_numpy(topk).cuda()
    offs, tok, rop = hz.group(d)
    o_offs, o_tok, o_rop = oracle.group_rows(topk, E)
    assert np.array_equal(offs.cpu().numpy(), o_offs)
    assert np.array_equal(tok.cpu().numpy(), o_tok)
    assert np.array_equal(rop.cpu().numpy(), o_rop)


def test_group_rows_bad_id_sets_status():
    import torch
    topk = np.array([[0, 5], [1, -1], [2, 0]], np.int32)
    p = hz.Problem(np.zeros((3, 8), np.uint16), np.zeros((4, 4, 1), np.uint32),
                   None, None, None, topk)
    d = hz.DeviceProblem(p, None, None)
    d.topk = torch.from_numpy(topk).cuda()
    offs, tok, rop = hz.group(d)
    assert q.q4moe_device_status(clear=True) & q.DEV_BAD_EXPERT_ID
    assert list(offs.cpu().numpy()) == [0, 2, 3, 4, 4]
    assert list(rop.cpu().numpy()) == [0, -1, 2, -1, 3, 1]


def test_group_rows_many_blocks_bad_ids():
    """Ids outside [0, E) on the many-block path: the status bit is set and
    those pairs get row -1; the others are a stable sort by expert."""
    import torch
    T, k, E = 4096, 4, 64
    topk = np.random.default_rng(5).integers(0, E, size=(T, k)).astype(
        np.int32)
    topk[7, 1] = E + 3
    topk[2000, 0] = -2
    p = hz.Problem(np.zeros((T, 8), np.uint16), np.zeros((E, 4, 1), np.uint32),
                   None, None, None, topk)
    d = hz.DeviceProblem(p, None, None)
    d.topk = torch.from_numpy(topk).cuda()
    q.q4moe_device_status(clear=True)
    offs, tok, rop = hz.group(d)
    assert q.q4moe_device_status(clear=True) & q.DEV_BAD_EXPERT_ID
    ids = topk.ravel()
    valid = [(int(e), qq) for qq, e in enumerate(ids) if 0 <= e < E]
    order = sorted(valid)                 # by expert, then pair index
    want_rop = np.full(ids.size, -1, np.int32)
    for row, (_, qq) in enumerate(order):
        want_rop[qq] = row
    want_offs = np.searchsorted([e for e, _ in order], np.arange(E + 1))
    assert np.array_equal(offs.cpu().numpy(), want_offs)
    assert np.array_equal(rop.cpu().numpy(), want_rop)
    assert np.array_equal(tok.cpu().numpy()[:len(order)],
                          np.array([qq // k for _, qq in order], np.int32))


# --------------------------------------------------------------------- tail --

def test_tail_exhaustive_bf16():
    """All 65,536 bf16 gate values (finite), several up values: the device
    tail equals the oracle's bit for bit (sigmoid, silu and out), and so
    does the sigmoid as the decode kernels form it (in registers when the
    fast form is conclusive, else from the table)."""
    import torch
    g = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    g = g[((g >> 7) & 0xFF) != 0xFF]
    for up in (1.0, -3.0, 0.0078125, 250.0):
        u = np.full(g.shape, syn.f32_to_bf16_bits(np.float32([up]))[0],
                    np.uint16)
        gd = torch.from_numpy(g.view(np.int16)).cuda()
        ud = torch.from_numpy(u.view(np.int16)).cuda()
        res = torch.empty((g.size, 4), dtype=torch.int16, device="cuda")
        q.q4moe_debug_tail(gd, ud, g.size, res)
        r = res.cpu().numpy().view(np.uint16)
        gf = syn.bf16_bits_to_f32(g)
        uf = syn.bf16_bits_to_f32(u)
        t = oracle.tail_array(gf, uf)
        bad = np.flatnonzero(r[:, 3] != t[:, 2])
        assert bad.size == 0, f"decode-form sigmoid: {bad.size} differ"
        for col, name in ((0, "sigmoid"), (1, "silu"), (2, "out")):
            bad = np.flatnonzero(r[:, col] != t[:, col + 2])
            assert bad.size == 0, f"{name}: {bad.size} differ, e.g. gate " \
                f"{g[bad[:4]]}"


# ------------------------------------------------------- exact integer data --

KERNELS = [q.KERNEL_AUTO, q.KERNEL_MATVEC, q.KERNEL_GEMM]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("E,I,H,T,k", [(1, 256, 512, 1, 1),
                                       (6, 128, 5120, 9, 3),
                                       (2, 384, 1024, 300, 2),
                                       (3, 36, 24, 7, 2)])
def test_exact_integer_bit_exact(kernel, E, I, H, T, k):
    p = hz.exact_problem(100 + H, E, I, H, T, k)
    if kernel == q.KERNEL_GEMM and (H % 64 or I % 128):
        with pytest.raises(q.Q4moeError):
            _run_and_compare(p, kernel=kernel, exact=True)
        return
    _run_and_compare(p, kernel=kernel, exact=True)


@pytest.mark.parametrize("kernel", KERNELS)
def test_exact_integer_ragged_counts(kernel):
    counts = [0, 1, 7, 8, 9, 47, 48, 49, 64, 65, 130, 0, 3]
    p = hz.problem_with_counts(5, counts, 256, 512, exact=True)
    _run_and_compare(p, kernel=kernel, exact=True)


# ----------------------------------------------------- real-valued parity --

def test_parity_single_expert_small_workload():
    """The 1-expert H=512 I=256 one-token workload, seed 0, all outputs."""
    w = syn.WORKLOADS["expert1_h512_i256_m1"]
    g = syn.generate(w)
    p = hz.Problem(g["x"], g["gate_w"], g["up_w"], g["gate_s"], g["up_s"],
                   g["topk"])
    _run_and_compare(p)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("E,T,k,routing,x_std", [
    (16, 12, 8, "uniform", 1.0),      # grouped decode shape, fewer experts
    (20, 40, 8, "zipf", 1.0),         # skewed verify shape
    (4, 96, 2, "uniform", 0.5),       # prefill-like rows per expert
])
def test_parity_reduced_workloads(kernel, E, T, k, routing, x_std):
    p = hz.random_problem(7 + T, E, 1536, 5120, T, k, routing, x_std)
    _run_and_compare(p, kernel=kernel)


@pytest.mark.parametrize("big", [13, 12])
def test_auto_mixes_matvec_and_gemm(big):
    """Automatic choice with I = 1536 (12 GEMM tiles per expert chunk): the
    experts above 16 rows (60, 48 and 17 rows) go to the GEMM while the
    small ones (1, 8, 9 rows, and an empty one) stay on the matvec.  The
    oracle's results, bit for bit on exact inputs."""
    counts = [60] * big + [1, 8, 9, 48, 0, 17]
    p = hz.problem_with_counts(80 + big, counts, 1536, 512, exact=True)
    _run_and_compare(p, exact=True)
    p = hz.problem_with_counts(90 + big, counts, 1536, 512)
    _run_and_compare(p)


@pytest.mark.parametrize("counts,launches", [([3] * 20, 1),
                                             ([60] + [1] * 39, 1),
                                             ([8] * 10, 2),
                                             ([60] * 2 + [1] * 6, 2),
                                             ([130, 129, 131], 1),
                                             ([200, 10, 200], 1)])
def test_auto_skips_a_gemm_that_cannot_get_work(counts, launches):
    """Under the automatic choice the GEMM is launched only when the call
    has at least 4 rows per expert: 60 rows over 20 experts, or 99 over 40
    with one expert of 60, take the matvec alone (one launch); 80 rows over
    10 experts launch the GEMM as well, which finds no expert above 16 rows;
    126 over 8 give it the two experts of 60.  From 128 rows per expert on
    average the GEMM alone takes every expert (one launch), a 10-row
    expert included.  Same results either way."""
    import torch
    p = hz.problem_with_counts(77, counts, 1536, 512, exact=True)
    d = hz.upload(p)
    offs_d, tok_d, _ = hz.group(d)
    torch.cuda.synchronize()
    n0 = q.q4moe_launch_count()
    gpu = hz.gate_up(d, offs_d, tok_d, debug=False)
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert q.q4moe_launch_count() - n0 == launches
    orc = _oracle_full(p, offs_d.cpu().numpy(), tok_d.cpu().numpy())
    assert np.array_equal(gpu["out"], orc["out"])


@pytest.mark.parametrize("counts", [[0, 1, 7, 8, 9, 47, 48, 49, 63, 64, 65,
                                     129, 200, 257]])
def test_parity_ragged_rows_per_expert(counts):
    p = hz.problem_with_counts(9, counts, 256, 512)
    for kernel in KERNELS:
        _run_and_compare(p, kernel=kernel)


@pytest.mark.parametrize("tile", [16, 32, 64, 128])
def test_matvec_tiles_bit_exact(tile):
    """Every unit height of the TMA-fed matvec, with I not a multiple of
    the tile (rows past I arrive as zeros and are never stored) and chunks
    of 1..8 rows."""
    counts = [0, 1, 7, 8, 9, 3, 16, 48, 2]
    p = hz.problem_with_counts(40 + tile, counts, 208, 1024, exact=True)
    _run_and_compare(p, kernel=q.KERNEL_MATVEC, exact=True, matvec_tile=tile)


@pytest.mark.parametrize("tile", [16, 32, 64, 128])
def test_matvec_tiles_real_valued(tile):
    p = hz.problem_with_counts(60 + tile, [1, 5, 8, 9, 0, 2], 1536, 5120)
    _run_and_compare(p, kernel=q.KERNEL_MATVEC, matvec_tile=tile)


@pytest.mark.parametrize("H", [384, 640])
def test_matvec_cp_async_path_base_mode(H):
    """H % 256 == 128 with slabs at base + e * stride: the matvec whose
    weights move by per-thread cp.async."""
    p = hz.problem_with_counts(H, [2, 0, 9, 1, 16], 96, H, exact=True)
    _run_and_compare(p, kernel=q.KERNEL_MATVEC, exact=True)
    p = hz.problem_with_counts(H + 1, [2, 0, 9, 1, 16], 96, H)
    _run_and_compare(p, kernel=q.KERNEL_MATVEC)


def _scale_bf16(x, shift):
    """bf16 bits times 2^shift (exponent field moved; zeros kept)."""
    x = x.astype(np.int32)
    nz = (x & 0x7FFF) != 0
    x[nz] += shift << 7
    return x.astype(np.uint16)


@pytest.mark.parametrize("shift", [40, -60, -90])
def test_matvec_scaled_exact_activations(shift):
    """Exact-integer activations times 2^shift.  The matvec stages a chunk
    of activations in f16 under a power-of-two scale when one fits (shift
    40 and -60), else in bf16 (-90: the scale would leave f32's range);
    every sum stays exact, so the bits must match the oracle's."""
    p = hz.problem_with_counts(77, [5, 8, 1, 3], 128, 512, exact=True)
    p.x = _scale_bf16(p.x, shift)
    _run_and_compare(p, kernel=q.KERNEL_MATVEC, exact=True)


def test_matvec_wide_exponent_span_falls_back_to_bf16():
    """Two rows of one chunk 2^40 apart (too wide a span for f16 under one
    scale) next to an ordinary chunk: bits must still match exactly."""
    p = hz.problem_with_counts(78, [2, 3], 128, 512, exact=True)
    rows = np.flatnonzero(p.topk[:, 0] == 0)
    p.x[rows[0]] = _scale_bf16(p.x[rows[0]][None], 20)[0]
    p.x[rows[1]] = _scale_bf16(p.x[rows[1]][None], -20)[0]
    _run_and_compare(p, kernel=q.KERNEL_MATVEC, exact=True)


def test_matvec_subnormal_activation_falls_back_to_bf16():
    p = hz.problem_with_counts(79, [3, 2], 256, 1024)
    p.x[0, 5] = 0x0001                     # smallest positive bf16 subnormal
    p.x[1, 7] = 0x8003
    _run_and_compare(p, kernel=q.KERNEL_MATVEC)


@pytest.mark.parametrize("exact", [True, False])
def test_gemm_with_and_without_token_count(exact):
    """The GEMM's tensor map over x spans num_tokens rows when the caller
    gives it, else the largest row count a coordinate can name; both must
    give the oracle's results."""
    p = hz.problem_with_counts(13, [70, 130, 3], 256, 512, exact=exact)
    _run_and_compare(p, kernel=q.KERNEL_GEMM, exact=exact)
    d = hz.upload(p)
    offs, tok, _ = hz.group(d)
    with_t = hz.gate_up(d, offs, tok, kernel=q.KERNEL_GEMM, debug=False)
    import torch
    M = int(tok.shape[0])
    out = torch.full((M, p.I), -1, dtype=torch.int16, device="cuda")
    o = q.q4moe_options_t()
    o.kernel = q.KERNEL_GEMM                # num_tokens left at 0
    q.q4moe_gate_up_swiglu_ex(d.x, d.slabs, offs, tok, M, p.H, p.I, out, o)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint16), with_t["out"])


def test_gemm_bad_token_row_reads_zeros():
    """A token index past num_tokens in a GEMM tile: the status bit is set
    and that row is computed from zero activations (output +0)."""
    import torch
    p = hz.problem_with_counts(14, [100], 256, 512)
    d = hz.upload(p)
    offs, tok, _ = hz.group(d)
    bad = tok.clone()
    bad[17] = p.T + 3
    q.q4moe_device_status(clear=True)
    res = hz.gate_up(d, offs, bad, kernel=q.KERNEL_GEMM)
    assert q.q4moe_device_status(clear=True) == q.DEV_BAD_TOKEN
    assert np.all(res["out"][17] == 0)
    assert np.all(res["gate32"][17] == 0) and np.all(res["up32"][17] == 0)
    good = hz.gate_up(d, offs, tok, kernel=q.KERNEL_GEMM)
    rows = np.arange(tok.shape[0]) != 17
    assert np.array_equal(res["out"][rows], good["out"][rows])


def test_parity_generic_shapes():
    """H not a multiple of 32 and tiny I (the pages' minimum rules)."""
    for (I, H) in ((4, 8), (12, 24), (20, 40)):
        p = hz.random_problem(I, 3, I, H, 5, 2)
        _run_and_compare(p)


def test_parity_noncanonical_layout_and_pointer_table():
    p = hz.random_problem(17, 5, 256, 512, 6, 2)
    I, H = p.I, p.H
    wb = I * H // 2
    L = q.q4moe_layout_t()
    L.hidden_size, L.intermediate_size = H, I
    # scales first, then up, then gate, with gaps
    L.up_s_offset = 0
    L.gate_s_offset = 4096
    L.up_w_offset = 8192
    L.gate_w_offset = 8192 + wb + 256
    L.slab_bytes = (L.gate_w_offset + wb + 4095) // 4096 * 4096
    _run_and_compare(p, layout=L, stride_pad=8192)
    _run_and_compare(p, ptr_table=True)
    _run_and_compare(p, kernel=q.KERNEL_GEMM, layout=L, stride_pad=8192)
    _run_and_compare(p, kernel=q.KERNEL_GEMM, ptr_table=True)
    # weight sections 16 bytes past a 32-byte boundary: the tensor-core
    # GEMM whose weight loads are 32 bytes wide is not taken, the other
    # one (with or without the workspace) gives the same results
    L16 = q.q4moe_layout_t()
    L16.hidden_size, L16.intermediate_size = H, I
    L16.up_s_offset = 0
    L16.gate_s_offset = 4096
    L16.up_w_offset = 8192 + 16
    L16.gate_w_offset = 8192 + 16 + wb + 256
    L16.slab_bytes = (L16.gate_w_offset + wb + 4095) // 4096 * 4096
    _run_and_compare(p, kernel=q.KERNEL_GEMM, layout=L16, stride_pad=8192)


def test_max_experts_and_empty_call():
    import torch
    p = hz.random_problem(3, q.MAX_EXPERTS, 8, 64, 70, 3)
    _run_and_compare(p)
    d = hz.upload(p)
    offs = torch.zeros(p.E + 1, dtype=torch.int32, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")[:0]
    out = torch.full((1, p.I), 7, dtype=torch.int16, device="cuda")
    q.q4moe_gate_up_swiglu(d.x, d.slabs, offs, tok, 0, p.H, p.I, out)
    torch.cuda.synchronize()
    assert torch.all(out == 7)          # M = 0 writes nothing


# ------------------------------------------------------ device-side checks --

def test_bad_offsets_and_tokens_raise_status():
    import torch
    p = hz.random_problem(4, 3, 16, 64, 4, 2)
    d = hz.upload(p)
    offs, tok, _ = hz.group(d)
    q.q4moe_device_status(clear=True)
    bad = offs.clone()
    bad[1] = bad[2] + 1                     # decreasing
    out = torch.full((8, p.I), 5, dtype=torch.int16, device="cuda")
    q.q4moe_gate_up_swiglu(d.x, d.slabs, bad, tok, 8, p.H, p.I, out)
    assert q.q4moe_device_status(clear=True) == q.DEV_BAD_ROW_OFFSETS
    assert torch.all(out == 5)              # nothing written
    badtok = tok.clone()
    badtok[3] = p.T + 5
    hz.gate_up(d, offs, badtok)             # num_tokens = T: checked
    assert q.q4moe_device_status(clear=True) == q.DEV_BAD_TOKEN


@pytest.mark.parametrize("counts", [[5], [3, 0, 6]])
def test_bad_offsets_tma_matvec_writes_nothing(counts):
    """The TMA matvec with inconsistent offsets: a single expert's call has
    already staged activations and issued weight loads when the offsets are
    checked; it must drain them, write nothing and raise the status bit."""
    import torch
    p = hz.problem_with_counts(11, counts, 256, 512)
    d = hz.upload(p)
    offs, tok, _ = hz.group(d)
    M = int(tok.shape[0])
    q.q4moe_device_status(clear=True)
    bad = offs.clone()
    bad[-1] = M + 1                           # last offset must be M
    out = torch.full((M, p.I), 5, dtype=torch.int16, device="cuda")
    o = q.q4moe_options_t()
    o.kernel = q.KERNEL_MATVEC
    q.q4moe_gate_up_swiglu_ex(d.x, d.slabs, bad, tok, M, p.H, p.I, out, o)
    assert q.q4moe_device_status(clear=True) == q.DEV_BAD_ROW_OFFSETS
    assert torch.all(out == 5)
    # the library still works afterwards
    _run_and_compare(p, kernel=q.KERNEL_MATVEC)


@pytest.mark.parametrize("exact", [True, False])
def test_single_expert_several_chunks(exact):
    """One expert, 20 rows: three chunks of activations, units computed
    before the offsets are read."""
    p = hz.problem_with_counts(12, [20], 1536, 4096, exact=exact)
    _run_and_compare(p, kernel=q.KERNEL_MATVEC, exact=exact)
    _run_and_compare(p, exact=exact)


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("I,H", [(100, 96), (1536, 4128), (256, 512)])
def test_single_expert_latency_kernel_shapes(M, I, H):
    """One expert with 1 to 8 rows runs on the kernel laid out for latency
    (each CTA ceil(I / SMs) intermediate rows, the K range split over its
    warps): K = 96 and 4128 (not multiples of 256, which the ring matvec
    needs), I = 100 (one row per CTA), row counts of each of its template
    sizes and between; exact and real-valued against the oracle."""
    for exact in (True, False):
        p = hz.problem_with_counts(40 + M + I, [M], I, H, exact=exact)
        _run_and_compare(p, exact=exact)


@pytest.mark.parametrize("shift", [40, -60, -90])
def test_single_expert_latency_kernel_scaled_activations(shift):
    """The latency kernel multiplies bf16 activations as they are (no f16
    staging): exact-integer activations times 2^shift still give exact
    sums, so the bits must match the oracle's."""
    p = hz.problem_with_counts(81, [3], 1536, 1024, exact=True)
    p.x = _scale_bf16(p.x, shift)
    _run_and_compare(p, exact=True)


@pytest.mark.parametrize("kernel", [q.KERNEL_AUTO, q.KERNEL_MATVEC])
def test_single_chunk_bad_token_reads_zeros(kernel):
    """One expert, 6 rows (a single chunk, whose rows of x move as bulk
    copies): a token index past num_tokens sets the status bit and its row
    is computed from zeros; the other rows are the oracle's."""
    p = hz.problem_with_counts(15, [6], 256, 1024, exact=True)
    d = hz.upload(p)
    offs, tok, _ = hz.group(d)
    bad = tok.clone()
    bad[2] = p.T + 1
    q.q4moe_device_status(clear=True)
    res = hz.gate_up(d, offs, bad, kernel=kernel)
    assert q.q4moe_device_status(clear=True) == q.DEV_BAD_TOKEN
    assert np.all(res["out"][2] == 0) and np.all(res["gate32"][2] == 0)
    good = hz.gate_up(d, offs, tok, kernel=kernel)
    rows = np.arange(6) != 2
    assert np.array_equal(res["out"][rows], good["out"][rows])
    _run_and_compare(p, kernel=kernel, exact=True)


def test_misaligned_slab_pointer_raises_status():
    import torch
    p = hz.random_problem(8, 2, 16, 64, 3, 1)
    d = hz.upload(p, ptr_table=True)
    ptrs = d.keep[-1]
    ptrs[1] += 64                            # no longer 4096-aligned
    offs, tok, _ = hz.group(d)
    hz.gate_up(d, offs, tok)
    assert q.q4moe_device_status(clear=True) & q.DEV_BAD_SLAB_PTR
    del torch


# ------------------------------------------------------ stream, determinism --

def test_side_stream_and_repeatability():
    import torch
    p = hz.random_problem(12, 8, 256, 1024, 20, 4)
    d = hz.upload(p)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        offs, tok, _ = hz.group(d, stream=s)
        a = hz.gate_up(d, offs, tok, stream=s)
        b = hz.gate_up(d, offs, tok, stream=s)
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(a["gate32"], b["gate32"])
