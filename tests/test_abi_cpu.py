"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before any CUDA
call (validation rules: page 52 validateCall, page 51 validateRange)."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

from up_swiglu_gb300 import q4moe as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "q4moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(q4moe_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = q.load()
    declared = _declared()
    assert declared, "no declarations parsed"
    assert sorted(q.EXPORTS) == declared
    for name in declared:
        assert hasattr(lib, name), name
    assert q.q4moe_abi_version() == q.ABI_VERSION


def test_canonical_layout():
    L = q.q4moe_canonical_layout(5120, 1536)
    assert (L.gate_w_offset, L.up_w_offset) == (0, 1536 * 2560)
    assert L.gate_s_offset == 1536 * 5120
    assert L.up_s_offset == 1536 * 5120 + 4 * 1536
    # down words after the up scales, rounded up to 256; down scales after
    # the down words; the slab rounded up to 4096
    assert L.down_w_offset == 7876608
    assert L.down_s_offset == 7876608 + 5120 * 768
    assert L.slab_bytes == 11829248 == 2888 * 4096
    L2 = q.q4moe_canonical_layout(512, 256)
    assert (L2.down_w_offset, L2.down_s_offset, L2.slab_bytes) == \
        (133120, 198656, 200704)
    assert q.q4moe_canonical_layout(4096, 1536).slab_bytes == 9465856
    L3 = q.q4moe_canonical_layout(64, 12)       # I % 8 != 0: no down
    assert (L3.down_w_offset, L3.down_s_offset) == (-1, -1)
    assert L3.slab_bytes == 4096
    L4 = q.q4moe_canonical_layout(64, 40)       # 8*I not a multiple of 256
    assert L4.down_w_offset == (2 * 40 * 32 + 8 * 40 + 255) // 256 * 256
    for H, I in ((0, 4), (12, 4), (8, 6), (8, 0), (-8, 4)):
        with pytest.raises(q.Q4moeError) as ei:
            q.q4moe_canonical_layout(H, I)
        assert ei.value.code == q.ERR_INVALID_ARG


def test_validate_layout_ranges_and_alignment():
    L = q.q4moe_canonical_layout(64, 8)
    q.q4moe_validate_layout(L)
    bad = q.q4moe_layout_t.from_buffer_copy(L)
    bad.up_s_offset = L.slab_bytes - 4          # runs past the slab
    with pytest.raises(q.Q4moeError) as ei:
        q.q4moe_validate_layout(bad)
    assert ei.value.code == q.ERR_RANGE
    bad = q.q4moe_layout_t.from_buffer_copy(L)
    bad.gate_s_offset = -4
    with pytest.raises(q.Q4moeError) as ei:
        q.q4moe_validate_layout(bad)
    assert ei.value.code == q.ERR_RANGE
    bad = q.q4moe_layout_t.from_buffer_copy(L)
    bad.gate_s_offset += 2
    with pytest.raises(q.Q4moeError) as ei:
        q.q4moe_validate_layout(bad)
    assert ei.value.code == q.ERR_ALIGNMENT


def test_canonical_layout_q8_and_packing():
    H, I = 64, 12
    L = q.q4moe_canonical_layout_format(H, I, q.FORMAT_Q8)
    assert L.weight_format == q.FORMAT_Q8
    assert (L.gate_w_offset, L.up_w_offset) == (0, I * H)
    assert (L.gate_s_offset, L.up_s_offset) == (2 * I * H, 2 * I * H + 4 * I)
    assert L.down_w_offset == (2 * I * H + 8 * I + 255) // 256 * 256
    assert L.down_s_offset == L.down_w_offset + H * I
    assert L.slab_bytes == 4096
    assert q.q4moe_canonical_layout_format(5120, 1536, q.FORMAT_Q8) \
        .slab_bytes == (2 * 1536 * 5120 + 8 * 1536 + 5120 * 1536 + 4 * 5120
                        + 4095) // 4096 * 4096
    rng = np.random.default_rng(1)
    gw = rng.integers(-128, 128, size=(I, H)).astype(np.int8)
    uw = rng.integers(-128, 128, size=(I, H)).astype(np.int8)
    dw = rng.integers(-128, 128, size=(H, I)).astype(np.int8)
    gs, us, ds = (rng.random(n).astype(np.float32) for n in (I, I, H))
    slab = np.full(L.slab_bytes, 0xAB, np.uint8)
    q.q4moe_pack_slab(L, gw, uw, gs, us, slab)
    q.q4moe_pack_slab_down(L, dw, ds, slab)
    assert np.array_equal(slab[:I * H].view(np.int8).reshape(I, H), gw)
    assert np.array_equal(slab[I * H:2 * I * H].view(np.int8).reshape(I, H),
                          uw)
    assert np.array_equal(slab[L.down_w_offset:L.down_w_offset + H * I]
                          .view(np.int8).reshape(H, I), dw)
    assert np.array_equal(slab[L.down_s_offset:L.down_s_offset + 4 * H]
                          .view(np.float32), ds)
    for H2, I2 in ((6, 4), (8, 6)):               # not multiples of 4
        with pytest.raises(q.Q4moeError):
            q.q4moe_canonical_layout_format(H2, I2, q.FORMAT_Q8)
    with pytest.raises(q.Q4moeError):
        q.q4moe_canonical_layout_format(64, 8, 7)   # unknown format
    bad = q.q4moe_layout_t.from_buffer_copy(L)
    bad.weight_format = 2
    with pytest.raises(q.Q4moeError):
        q.q4moe_validate_layout(bad)
    # a Q4 layout read as Q8 needs twice the weight bytes: the down words
    # run past the slab
    bad = q.q4moe_layout_t.from_buffer_copy(
        q.q4moe_canonical_layout(5120, 1536))
    bad.weight_format = q.FORMAT_Q8
    with pytest.raises(q.Q4moeError) as ei:
        q.q4moe_validate_layout(bad)
    assert ei.value.code == q.ERR_RANGE


def test_validate_layout_down_sections():
    L = q.q4moe_canonical_layout(64, 8)
    bad = q.q4moe_layout_t.from_buffer_copy(L)
    bad.down_s_offset = -1                      # one of the two absent
    with pytest.raises(q.Q4moeError) as ei:
        q.q4moe_validate_layout(bad)
    assert ei.value.code == q.ERR_INVALID_ARG
    bad = q.q4moe_layout_t.from_buffer_copy(L)
    bad.down_s_offset = L.slab_bytes - 4 * 64 + 4   # past the slab
    with pytest.raises(q.Q4moeError) as ei:
        q.q4moe_validate_layout(bad)
    assert ei.value.code == q.ERR_RANGE
    bad = q.q4moe_layout_t.from_buffer_copy(L)
    bad.down_w_offset += 2
    with pytest.raises(q.Q4moeError) as ei:
        q.q4moe_validate_layout(bad)
    assert ei.value.code == q.ERR_ALIGNMENT
    no_down = q.q4moe_layout_t.from_buffer_copy(L)
    no_down.down_w_offset = no_down.down_s_offset = -1
    q.q4moe_validate_layout(no_down)
    with pytest.raises(q.Q4moeError):
        q.q4moe_pack_slab_down(no_down, np.zeros(64, np.uint32),
                               np.zeros(64, np.float32),
                               np.zeros(L.slab_bytes, np.uint8))


def test_pack_slab_places_sections():
    H, I = 64, 8
    L = q.q4moe_canonical_layout(H, I)
    rng = np.random.default_rng(0)
    gw = rng.integers(0, 2**32, size=(I, H // 8), dtype=np.uint64).astype(
        np.uint32)
    uw = rng.integers(0, 2**32, size=(I, H // 8), dtype=np.uint64).astype(
        np.uint32)
    gs = rng.random(I).astype(np.float32)
    us = rng.random(I).astype(np.float32)
    slab = np.full(L.slab_bytes, 0xAB, np.uint8)
    q.q4moe_pack_slab(L, gw, uw, gs, us, slab)
    wb = I * H // 2
    assert np.array_equal(slab[:wb].view(np.uint32).reshape(I, -1), gw)
    assert np.array_equal(slab[wb:2 * wb].view(np.uint32).reshape(I, -1), uw)
    assert np.array_equal(slab[2 * wb:2 * wb + 4 * I].view(np.float32), gs)
    assert np.array_equal(
        slab[2 * wb + 4 * I:2 * wb + 8 * I].view(np.float32), us)
    assert np.all(slab[2 * wb + 8 * I:] == 0)
    dw = rng.integers(0, 2**32, size=(H, I // 8), dtype=np.uint64).astype(
        np.uint32)
    ds = rng.random(H).astype(np.float32)
    q.q4moe_pack_slab_down(L, dw, ds, slab)
    d0, s0 = L.down_w_offset, L.down_s_offset
    assert np.array_equal(slab[d0:d0 + H * I // 2].view(np.uint32)
                          .reshape(H, -1), dw)
    assert np.array_equal(slab[s0:s0 + 4 * H].view(np.float32), ds)
    assert np.array_equal(slab[:wb].view(np.uint32).reshape(I, -1), gw)
    assert np.all(slab[2 * wb + 8 * I:d0] == 0)
    assert np.all(slab[s0 + 4 * H:] == 0)


FAKE = 1 << 40     # an aligned address that is never dereferenced on host


def _call(x=FAKE, slabs=None, offs=FAKE, tok=FAKE, M=4, H=64, I=8,
          out=FAKE, opts=None):
    lib = q.load()
    L = q.q4moe_canonical_layout(64, 8)
    s = slabs if slabs is not None else q.make_slabs(2, L, base=FAKE)
    return lib.q4moe_gate_up_swiglu_ex(
        x, ctypes.byref(s) if s is not False else None, offs, tok, M, H, I,
        out, None if opts is None else ctypes.byref(opts), None)


def test_host_argument_errors():
    L = q.q4moe_canonical_layout(64, 8)
    assert _call(slabs=False) == q.ERR_INVALID_ARG
    assert _call(H=128) == q.ERR_INVALID_ARG               # differs from layout
    assert _call(M=-1) == q.ERR_INVALID_ARG
    assert _call(offs=None) == q.ERR_INVALID_ARG
    assert _call(x=None) == q.ERR_INVALID_ARG
    assert _call(x=FAKE + 8) == q.ERR_ALIGNMENT            # x not 16-aligned
    assert _call(slabs=q.make_slabs(2, L, base=FAKE + 64)) == \
        q.ERR_ALIGNMENT
    assert _call(slabs=q.make_slabs(2, L, base=FAKE,
                                    slab_stride=4100)) == q.ERR_ALIGNMENT
    assert _call(slabs=q.make_slabs(0, L, base=FAKE)) == q.ERR_INVALID_ARG
    assert _call(slabs=q.make_slabs(q.MAX_EXPERTS + 1, L, base=FAKE)) == \
        q.ERR_INVALID_ARG
    bad = q.q4moe_layout_t.from_buffer_copy(L)
    bad.up_w_offset = L.slab_bytes
    assert _call(slabs=q.make_slabs(2, bad, base=FAKE)) == q.ERR_RANGE
    o = q.q4moe_options_t()
    o.kernel = 7
    assert _call(opts=o) == q.ERR_INVALID_ARG
    assert "options" in q.q4moe_last_error()
    o = q.q4moe_options_t()
    o.workspace = FAKE
    o.workspace_bytes = q.q4moe_workspace_bytes(4, 64) - 1
    assert _call(opts=o) == q.ERR_INVALID_ARG       # workspace too small
    o.workspace = FAKE + 16
    o.workspace_bytes = 1 << 20
    assert _call(opts=o) == q.ERR_ALIGNMENT         # not 256-aligned
    assert q.q4moe_workspace_bytes(4, 64) == 512
    assert q.q4moe_workspace_bytes(3, 8) == 256
    lib = q.load()
    assert lib.q4moe_group_rows(FAKE, 4, 0, 8, FAKE, FAKE, FAKE, None) == \
        q.ERR_INVALID_ARG
    assert lib.q4moe_group_rows(FAKE, 4, 2, q.MAX_EXPERTS + 1, FAKE, FAKE,
                                FAKE, None) == q.ERR_INVALID_ARG
    assert lib.q4moe_debug_tail(None, None, 4, None, None) == \
        q.ERR_INVALID_ARG
    assert lib.q4moe_debug_tail_mlx(None, None, 4, None, None) == \
        q.ERR_INVALID_ARG
    # the wait diagnostic takes limits of 1 us .. 1 s only
    for ns in (0, 999, 1000000001, -5):
        assert lib.q4moe_debug_wait_timeout(ns, None) == q.ERR_INVALID_ARG
    # the tail option: MLX's is for trellis codes only, values outside the
    # three and a nonzero reserved field are refused
    for tail, reserved in ((q.TAIL_MLX, 0), (3, 0), (-1, 0),
                           (q.TAIL_PAGE, 1)):
        o = q.q4moe_options_t()
        o.tail, o.reserved1 = tail, reserved
        assert _call(opts=o) == q.ERR_INVALID_ARG, (tail, reserved)
    o = q.q4moe_options_t()
    o.tail = q.TAIL_MLX
    assert _call(opts=o) == q.ERR_INVALID_ARG
    assert "MLX tail" in q.q4moe_last_error()


def test_down_and_mlp_host_argument_errors():
    lib = q.load()
    L = q.q4moe_canonical_layout(64, 8)
    s = q.make_slabs(2, L, base=FAKE)

    def down(mid=FAKE, slabs=s, offs=FAKE, M=4, H=64, I=8, out=FAKE,
             opts=None):
        return lib.q4moe_down_proj(mid, ctypes.byref(slabs), offs, M, H, I,
                                   out, None if opts is None
                                   else ctypes.byref(opts), None)

    def mlp(x=FAKE, mid=FAKE + (1 << 20), out=FAKE + (2 << 20), slabs=s,
            M=4):
        return lib.q4moe_expert_mlp(x, ctypes.byref(slabs), FAKE, FAKE, M, 64,
                                    8, mid, out, None, None)

    assert down(mid=FAKE + 8) == q.ERR_ALIGNMENT      # mid not 16-aligned
    assert down(out=FAKE + 1) == q.ERR_ALIGNMENT
    assert down(offs=None) == q.ERR_INVALID_ARG
    assert down(mid=None) == q.ERR_INVALID_ARG
    assert down(I=16) == q.ERR_INVALID_ARG            # differs from layout
    no_down = q.q4moe_layout_t.from_buffer_copy(L)
    no_down.down_w_offset = no_down.down_s_offset = -1
    nd = q.make_slabs(2, no_down, base=FAKE)
    assert down(slabs=nd) == q.ERR_INVALID_ARG
    assert "down sections" in q.q4moe_last_error()
    for field, val in (("num_tokens", 4), ("up_f32", FAKE),
                       ("workspace", FAKE), ("tail", q.TAIL_MLX)):
        o = q.q4moe_options_t()
        setattr(o, field, val)
        assert down(opts=o) == q.ERR_INVALID_ARG, field
    assert mlp(slabs=nd) == q.ERR_INVALID_ARG
    assert mlp(mid=FAKE + 8) == q.ERR_ALIGNMENT
    assert mlp(mid=FAKE + 64, out=FAKE) == q.ERR_INVALID_ARG   # overlap
    assert "overlaps" in q.q4moe_last_error()
    import torch
    if not torch.cuda.is_available():
        assert down() in (q.ERR_CUDA, q.ERR_DEVICE)
        assert mlp() in (q.ERR_CUDA, q.ERR_DEVICE)


def test_valid_call_without_gpu_reports_device_error():
    """A call that passes host validation needs a device: without one it
    returns a CUDA/device error instead of computing anything."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = _call()
    assert rc in (q.ERR_CUDA, q.ERR_DEVICE)


def test_trellis_layout_and_host_errors():
    """Trellis slabs: canonical section offsets (256-byte boundaries, size
    rounded to 4096), geometry checks, packing, and host argument errors of
    the trellis entry point (no GPU needed)."""
    H, I, T, L, kg, ku = 512, 40, 256, 12, 4, 3
    lay = q.q4moe_trellis_canonical_layout(H, I, T, L, kg, ku)
    gb, ub = I * H * kg // 8, I * H * ku // 8
    up256 = lambda v: (v + 255) // 256 * 256  # noqa: E731
    assert lay.gate_codes_offset == 0
    assert lay.up_codes_offset == up256(gb)
    assert lay.gate_scales_offset == up256(lay.up_codes_offset + ub)
    assert lay.up_scales_offset == up256(lay.gate_scales_offset + 2 * I)
    assert lay.slab_bytes % 4096 == 0
    assert lay.slab_bytes >= lay.up_scales_offset + 2 * I
    for args in ((H, I, 100, L, kg, ku),       # block not a multiple of 32
                 (H, I, 384, L, kg, ku),       # block does not divide H
                 (H, I, T, 25, kg, ku),        # window too wide
                 (H, I, T, L, 9, ku),          # width above 8
                 (H, 0, T, L, kg, ku)):
        with pytest.raises(q.Q4moeError):
            q.q4moe_trellis_canonical_layout(*args)
    rng = np.random.default_rng(2)
    gc = rng.integers(0, 2**32, size=(I, H * kg // 32),
                      dtype=np.uint64).astype(np.uint32)
    uc = rng.integers(0, 2**32, size=(I, H * ku // 32),
                      dtype=np.uint64).astype(np.uint32)
    gs = rng.integers(0, 2**16, size=I).astype(np.uint16)
    us = rng.integers(0, 2**16, size=I).astype(np.uint16)
    slab = np.full(lay.slab_bytes, 0xCD, np.uint8)
    q.q4moe_trellis_pack_slab(lay, gc, uc, gs, us, slab)
    assert np.array_equal(slab[:gb].view(np.uint32).reshape(I, -1), gc)
    o = lay.up_codes_offset
    assert np.array_equal(slab[o:o + ub].view(np.uint32).reshape(I, -1), uc)
    o = lay.up_scales_offset
    assert np.array_equal(slab[o:o + 2 * I].view(np.uint16), us)
    lib = q.load()
    s = q.make_trellis_slabs(2, lay, base=FAKE)

    def call(x=FAKE, slabs=s, M=4, Hc=H, opts=None):
        return lib.q4moe_trellis_gate_up_swiglu(
            x, ctypes.byref(slabs), FAKE, FAKE, M, Hc, I, FAKE,
            None if opts is None else ctypes.byref(opts), None)

    assert call(Hc=1024) == q.ERR_INVALID_ARG          # differs from layout
    assert call(x=FAKE + 8) == q.ERR_ALIGNMENT
    assert call(slabs=q.make_trellis_slabs(2, lay, base=FAKE + 64)) == \
        q.ERR_ALIGNMENT
    o = q.q4moe_options_t()
    o.kernel = q.KERNEL_GEMM
    assert call(opts=o) == q.ERR_INVALID_ARG           # no kernel choice
    o = q.q4moe_options_t()
    o.tail = 3
    assert call(opts=o) == q.ERR_INVALID_ARG           # no such tail
    bad = q.q4moe_trellis_layout_t.from_buffer_copy(lay)
    bad.up_scales_offset = lay.slab_bytes - 2
    assert call(slabs=q.make_trellis_slabs(2, bad, base=FAKE)) == \
        q.ERR_RANGE
    import torch
    if not torch.cuda.is_available():
        assert call() in (q.ERR_CUDA, q.ERR_DEVICE)
        for tail in (q.TAIL_AUTO, q.TAIL_PAGE, q.TAIL_MLX):
            o = q.q4moe_options_t()
            o.tail = tail                # accepted: fails only for the GPU
            assert call(opts=o) in (q.ERR_CUDA, q.ERR_DEVICE)
