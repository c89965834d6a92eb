"""The allocation-free entry point, q4moe_gate_up_swiglu_noalloc.

Some callers cannot allocate device memory (a plugin inside a host engine
that owns the GPU's memory, a fixed memory budget, a loop that must not risk
an allocator's device synchronisation); this entry point serves them with a
scratch array that lives inside the library.  Its results must match the
regular entry point's, call after call, although every call reuses the same
array.  This file is collected last so that a run stopping at the first
failure has run every other test already.
"""
from __future__ import annotations

import numpy as np
import pytest

import harness as hz
from up_swiglu_gb300 import q4moe as q

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    q.load()
    q.q4moe_device_status(clear=True)
    yield
    assert q.q4moe_device_status(clear=True) == 0


def _outputs(d, offs, tok, noalloc):
    """The no-alloc call, or the regular one given a workspace of its own
    (the same kernels and the same summation order)."""
    import torch
    M = int(tok.shape[0])
    out = torch.full((M, d.p.I), -1, dtype=torch.int16, device="cuda")
    if noalloc:
        q.q4moe_gate_up_swiglu_noalloc(d.x, d.slabs, offs, tok, M, d.p.H,
                                       d.p.I, out)
    else:
        ws = torch.empty(q.q4moe_workspace_bytes(M, d.p.H) + 256,
                         dtype=torch.uint8, device="cuda")
        o = q.q4moe_options_t()
        o.workspace = ws.data_ptr() + (-ws.data_ptr()) % 256
        o.workspace_bytes = q.q4moe_workspace_bytes(M, d.p.H)
        q.q4moe_gate_up_swiglu_ex(d.x, d.slabs, offs, tok, M, d.p.H, d.p.I,
                                  out, o)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16)


def _gemm_reference(d, offs, tok):
    """The regular entry point with the GEMM forced and a torch-allocated
    workspace: the path the no-alloc call takes with its own scratch."""
    import torch
    M = int(tok.shape[0])
    out = torch.full((M, d.p.I), -1, dtype=torch.int16, device="cuda")
    ws = torch.empty(q.q4moe_workspace_bytes(M, d.p.H) + 256,
                     dtype=torch.uint8, device="cuda")
    o = q.q4moe_options_t()
    o.kernel = q.KERNEL_GEMM
    off = (-ws.data_ptr()) % 256
    o.workspace = ws.data_ptr() + off
    o.workspace_bytes = q.q4moe_workspace_bytes(M, d.p.H)
    q.q4moe_gate_up_swiglu_ex(d.x, d.slabs, offs, tok, M, d.p.H, d.p.I, out,
                              o)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16)


def test_noalloc_gemm_path_uses_its_scratch_twice():
    """One expert with 1280 rows at I = 4096: 5 x 32 GEMM tiles fill every
    SM, so the automatic choice sends the call to the tensor-core GEMM, whose
    row copy writes the library's scratch (1280 x 512 x 2 bytes) and whose
    TMA loads read it back.  A different problem fills the scratch first;
    then two calls in a row must match the regular entry point with its own
    workspace bit for bit, each launching the row copy and the GEMM."""
    p0 = hz.problem_with_counts(77, [1280], 4096, 512)
    d0 = hz.upload(p0)
    offs0, tok0, _ = hz.group(d0)
    _outputs(d0, offs0, tok0, noalloc=True)      # other contents first
    p = hz.problem_with_counts(78, [1280], 4096, 512)
    d = hz.upload(p)
    offs, tok, _ = hz.group(d)
    want = _gemm_reference(d, offs, tok)
    for _ in range(2):
        n0 = q.q4moe_launch_count()
        got = _outputs(d, offs, tok, noalloc=True)
        assert q.q4moe_launch_count() - n0 == 2  # row copy + GEMM
        assert np.array_equal(got, want)


@pytest.mark.parametrize("counts,I,H", [
    ([0, 60, 130, 7, 257, 1, 90], 256, 512),      # matvec (automatic choice)
    ([3, 1, 8, 0, 2], 384, 1024),                 # matvec-only experts
])
def test_noalloc_matches_regular_entry_point_twice(counts, I, H):
    p = hz.problem_with_counts(31 + H, counts, I, H)
    d = hz.upload(p)
    offs, tok, _ = hz.group(d)
    want = _outputs(d, offs, tok, noalloc=False)
    # two calls in a row: the second finds the first call's scratch
    # contents and must not depend on them
    for _ in range(2):
        got = _outputs(d, offs, tok, noalloc=True)
        assert np.array_equal(got, want)
    # a second problem through the same scratch, then the first again
    p2 = hz.problem_with_counts(5, [200, 70], 256, 512)
    d2 = hz.upload(p2)
    offs2, tok2, _ = hz.group(d2)
    assert np.array_equal(_outputs(d2, offs2, tok2, noalloc=True),
                          _outputs(d2, offs2, tok2, noalloc=False))
    assert np.array_equal(_outputs(d, offs, tok, noalloc=True), want)


def test_noalloc_rejects_problems_beyond_its_scratch():
    import torch
    H = 8192
    M = q.NOALLOC_SCRATCH_BYTES // (2 * H) + 1       # one row too many
    L = q.q4moe_canonical_layout(H, 128)
    slabs = q.make_slabs(1, L, base=1 << 40)
    x = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.Q4moeError) as ei:
        q.q4moe_gate_up_swiglu_noalloc(x, slabs, x, x, M, H, 128, x)
    assert ei.value.code == q.ERR_INVALID_ARG
    assert "scratch" in str(ei.value)
