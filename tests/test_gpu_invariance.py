"""Batch invariance (Q4MOE_KERNEL_BATCH_INVARIANT): a row's output bits do
not depend on the other rows of the call.

Page 52 of "@mlx-bun/inference 0.0.0-stage -> 1.0.0" (streamed-experts.ts)
runs one SIMD group per output row and sample, so a row decoded alone and
the same row inside a speculative-verify batch agree bit for bit; the mode
keeps that property.  Each test computes rows inside a large call, then
alone (or in other company) and compares bits; the large call is also
checked against the oracle."""
from __future__ import annotations

import numpy as np
import pytest

import harness as hz
import oracle
import parity
from up_swiglu_gb300 import q4moe as q
from up_swiglu_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

INV = q.KERNEL_BATCH_INVARIANT


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


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _gate_up_rows(d, tokens, experts, E, kernel=INV, tile=0):
    """Call with grouped rows reading x rows `tokens`, expert `experts[j]`
    for row j (experts ascending); returns out bits [len, I]."""
    counts = np.bincount(experts, minlength=E)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return hz.gate_up(d, _dev(offs), _dev(np.asarray(tokens, np.int32)),
                      kernel=kernel, matvec_tile=tile, debug=False)["out"]


@pytest.mark.parametrize("ptr_table", [False, True])
def test_gate_up_row_alone_equals_row_in_batch(ptr_table):
    """Expert 0 with 200 rows, expert 1 with 1, expert 2 with 37 (H = 1024,
    I = 512): each of several rows, called alone, in a 2-row call and in the
    whole call, gives the same bits; the whole call matches the oracle.  One
    token has a value 2^40 times its neighbours, so its chunk stays in bf16
    while the others run in f16: the other rows of that chunk must still
    agree with their lone calls.  With a pointer table the generic kernel
    runs (same property)."""
    E, I, H = 3, 512, 1024
    T = 240
    p = hz.random_problem(5, E, I, H, T, 1)
    wide = 13
    xw = syn.bf16_bits_to_f32(p.x).copy()
    xw[wide, 5] = xw[wide, 5] * np.float32(2.0 ** 40)
    p.x = syn.f32_to_bf16_bits(xw)
    d = hz.upload(p, ptr_table=ptr_table)
    experts = np.array([0] * 200 + [1] + [2] * 37)
    tokens = np.arange(experts.size) % T
    full = _gate_up_rows(d, tokens, experts, E)
    offs = np.concatenate([[0], np.cumsum(np.bincount(experts, minlength=E))
                           ]).astype(np.int32)
    orc = oracle.gate_up_swiglu(p.x, p.gate_w, p.up_w, p.gate_s, p.up_s,
                                offs, tokens.astype(np.int32),
                                want_debug=True)
    gs, us = hz.element_scales(p, offs)
    gpu = hz.gate_up(d, _dev(offs), _dev(tokens.astype(np.int32)),
                     kernel=INV)
    assert np.array_equal(gpu["out"], full)
    parity.compare(gpu, orc, gs, us, H)
    for r in (0, 8, 12, 14, 15, 199, 200, 201, 237):
        alone = _gate_up_rows(d, [tokens[r]], [experts[r]], E)
        assert np.array_equal(alone[0], full[r]), r
        # the same row second in a pair, next to another token
        pair = _gate_up_rows(d, [tokens[(r + 3) % 200], tokens[r]],
                             [experts[r], experts[r]], E)
        assert np.array_equal(pair[1], full[r]), r


@pytest.mark.parametrize("tile", [16, 128])
def test_down_row_alone_equals_row_in_batch(tile):
    """The down projection in the same mode: every row of a 3-expert call
    equals the row computed alone (K = 1536, N = 512)."""
    import torch
    p, mid, offs = hz.down_only_problem(9, [70, 1, 9], 1536, 512)
    d = hz.upload(p)
    full = hz.down(d, offs, mid, kernel=INV, matvec_tile=tile)
    orc = oracle.down_proj(mid, p.down_w, p.down_s, offs, want_debug=True)
    parity.compare_down(full, orc, hz.down_scales(p, offs), 1536)
    e_of = np.repeat(np.arange(3), np.diff(offs))
    for r in (0, 7, 8, 69, 70, 71, 79):
        o1 = np.zeros(4, np.int32)
        o1[e_of[r] + 1:] = 1
        alone = hz.down(d, o1, mid[r:r + 1], kernel=INV, matvec_tile=tile,
                        debug=False)
        assert np.array_equal(alone["out"][0], full["out"][r]), r
    torch.cuda.synchronize()


def test_invariant_mode_on_exact_inputs_matches_the_oracle_bits():
    p = hz.exact_problem(21, 4, 256, 512, 300, 2)
    d = hz.upload(p)
    offs_d, tok_d, _ = hz.group(d)
    gpu = hz.gate_up(d, offs_d, tok_d, kernel=INV)
    orc = oracle.gate_up_swiglu(p.x, p.gate_w, p.up_w, p.gate_s, p.up_s,
                                offs_d.cpu().numpy(), tok_d.cpu().numpy(),
                                want_debug=True)
    gs, us = hz.element_scales(p, offs_d.cpu().numpy())
    parity.compare(gpu, orc, gs, us, p.H, exact=True)
