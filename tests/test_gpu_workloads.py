"""Full-size synthetic workloads on the GPU, in the launch configuration the
benchmark times (automatic kernel choice), checked against the oracle on
sampled outputs it computes one by one."""
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
    q.load()
    oracle.build()
    q.q4moe_device_status(clear=True)
    yield
    assert q.q4moe_device_status(clear=True) == 0


def _problem(name):
    w = syn.WORKLOADS[name]
    g = syn.generate(w)
    return w, hz.Problem(g["x"], g["gate_w"], g["up_w"], g["gate_s"],
                         g["up_s"], g["topk"])


def test_single_expert_decode_repeated():
    """H=4096, I=1536, one token: all outputs vs the oracle, and the call
    repeated 1000 times gives the same bits every time."""
    import torch
    w, p = _problem("expert1_h4096_i1536_m1_x1000")
    d = hz.upload(p)
    offs, tok, _ = hz.group(d)
    gpu = hz.gate_up(d, offs, tok)
    orc = oracle.gate_up_swiglu(p.x, p.gate_w, p.up_w, p.gate_s, p.up_s,
                                offs.cpu().numpy(), tok.cpu().numpy(),
                                want_debug=True)
    gs, us = hz.element_scales(p, offs.cpu().numpy())
    parity.compare(gpu, orc, gs, us, p.H)
    out = torch.empty((1, p.I), dtype=torch.int16, device="cuda")
    first = None
    for r in range(w.repeats):
        q.q4moe_gate_up_swiglu(d.x, d.slabs, offs, tok, 1, p.H, p.I, out)
        if r == 0:
            first = out.clone()
    torch.cuda.synchronize()
    assert torch.equal(out, first)
    assert np.array_equal(first.cpu().numpy().view(np.uint16), gpu["out"])


@pytest.mark.parametrize("name", ["moe128_top8_t32_h5120_i1536",
                                  "moe160_top8_t128_zipf_h5120_i1536",
                                  "moe160_top8_t4096_h5120_i1536"])
def test_full_size_sampled(name):
    w, p = _problem(name)
    d = hz.upload(p)
    offs_d, tok_d, rop_d = hz.group(d)
    offs, tok = offs_d.cpu().numpy(), tok_d.cpu().numpy()
    o_offs, o_tok, o_rop = oracle.group_rows(p.topk, p.E)
    assert np.array_equal(offs, o_offs) and np.array_equal(tok, o_tok)
    assert np.array_equal(rop_d.cpu().numpy(), o_rop)
    gpu = hz.gate_up(d, offs_d, tok_d)
    M, I = gpu["out"].shape
    assert M == w.routed_rows
    # properties at full size: every output and f32 value finite
    assert np.all(((gpu["out"] >> 7) & 0xFF) != 0xFF)
    assert np.all(np.isfinite(gpu["gate32"])) and np.all(
        np.isfinite(gpu["up32"]))
    # sampled elements: random ones plus every column of the first and last
    # grouped rows and of the busiest expert's first row
    rng = np.random.default_rng(M)
    rows = list(rng.integers(0, M, 3000))
    cols = list(rng.integers(0, I, 3000))
    busiest = int(np.argmax(np.diff(offs)))
    for r in (0, M - 1, int(offs[busiest])):
        rows += [r] * I
        cols += list(range(I))
    rows, cols = np.array(rows), np.array(cols)
    orc = oracle.gate_up_swiglu_sampled(p.x, p.gate_w, p.up_w, p.gate_s,
                                        p.up_s, offs, tok, rows, cols)
    gs_el, us_el = hz.element_scales(p, offs)
    sel = {k: gpu[k][rows, cols] for k in ("out", "gate32", "up32")}
    parity.compare(sel, orc, gs_el[rows, cols], us_el[rows, cols], p.H)
    # the plain entry point gives the same bits as the debug one, and so
    # does the call with a workspace (the benchmark's configuration)
    plain = hz.gate_up(d, offs_d, tok_d, debug=False)
    assert np.array_equal(plain["out"], gpu["out"])
    ws = hz.gate_up(d, offs_d, tok_d, debug=False, workspace=True)
    assert np.array_equal(ws["out"], gpu["out"])
