"""Python binding of libq4moe (include/q4moe.h): argument marshalling only.

The functions below carry the C names and arguments; tensors (torch) are
passed as device pointers, streams as ``torch.cuda.Stream`` or raw handles.
Every step of the computation runs in the library's CUDA kernels; there is
no CPU or PyTorch fallback, and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

ABI_VERSION = 8
SLAB_ALIGNMENT = 4096
MAX_EXPERTS = 1024

OK = 0
ERR_INVALID_ARG = -1
ERR_ALIGNMENT = -2
ERR_RANGE = -3
ERR_DEVICE = -4
ERR_CUDA = -5
ERR_DEVICE_DATA = -6

DEV_BAD_ROW_OFFSETS = 0x1
DEV_BAD_TOKEN = 0x2
DEV_BAD_SLAB_PTR = 0x4
DEV_BAD_EXPERT_ID = 0x8
DEV_WAIT_TIMEOUT = 0x10

FORMAT_Q4 = 0
FORMAT_Q8 = 1

KERNEL_AUTO = 0
KERNEL_MATVEC = 1
KERNEL_GEMM = 2
KERNEL_BATCH_INVARIANT = 3

# SwiGLU tail (q4moe_options_t.tail): AUTO = the pages' choice (page 52's,
# MLX's for trellis codes whose gate and up widths differ), PAGE = page 52's,
# MLX = MLX's compiled SwiGLU in bf16 arithmetic (trellis calls only).
TAIL_AUTO = 0
TAIL_PAGE = 1
TAIL_MLX = 2

# Every symbol include/q4moe.h declares (checked by the CPU tests).
EXPORTS = (
    "q4moe_abi_version", "q4moe_last_error", "q4moe_canonical_layout",
    "q4moe_validate_layout", "q4moe_pack_slab", "q4moe_group_rows",
    "q4moe_gate_up_swiglu", "q4moe_gate_up_swiglu_ex", "q4moe_device_status",
    "q4moe_debug_tail", "q4moe_launch_count", "q4moe_workspace_bytes",
    "q4moe_gate_up_swiglu_noalloc", "q4moe_pack_slab_down",
    "q4moe_down_proj", "q4moe_expert_mlp", "q4moe_canonical_layout_format",
    "q4moe_trellis_canonical_layout", "q4moe_trellis_pack_slab",
    "q4moe_trellis_gate_up_swiglu", "q4moe_debug_tail_mlx",
    "q4moe_debug_wait_timeout",
)

# Size of the library's fixed scratch used by q4moe_gate_up_swiglu_noalloc.
NOALLOC_SCRATCH_BYTES = 32 << 20


class Q4moeError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"q4moe error {code}: {message}")
        self.code = code


class q4moe_layout_t(ctypes.Structure):
    _fields_ = [("hidden_size", ctypes.c_int64),
                ("intermediate_size", ctypes.c_int64),
                ("slab_bytes", ctypes.c_int64),
                ("gate_w_offset", ctypes.c_int64),
                ("up_w_offset", ctypes.c_int64),
                ("gate_s_offset", ctypes.c_int64),
                ("up_s_offset", ctypes.c_int64),
                ("down_w_offset", ctypes.c_int64),
                ("down_s_offset", ctypes.c_int64),
                ("weight_format", ctypes.c_int64)]


class q4moe_slabs_t(ctypes.Structure):
    _fields_ = [("num_experts", ctypes.c_int32),
                ("reserved0", ctypes.c_int32),
                ("base", ctypes.c_void_p),
                ("slab_stride", ctypes.c_int64),
                ("slab_ptrs", ctypes.c_void_p),
                ("layout", q4moe_layout_t)]


class q4moe_trellis_layout_t(ctypes.Structure):
    _fields_ = [("hidden_size", ctypes.c_int64),
                ("intermediate_size", ctypes.c_int64),
                ("block_size", ctypes.c_int32),
                ("window_bits", ctypes.c_int32),
                ("gate_bits", ctypes.c_int32),
                ("up_bits", ctypes.c_int32),
                ("slab_bytes", ctypes.c_int64),
                ("gate_codes_offset", ctypes.c_int64),
                ("up_codes_offset", ctypes.c_int64),
                ("gate_scales_offset", ctypes.c_int64),
                ("up_scales_offset", ctypes.c_int64)]


class q4moe_trellis_slabs_t(ctypes.Structure):
    _fields_ = [("num_experts", ctypes.c_int32),
                ("reserved0", ctypes.c_int32),
                ("base", ctypes.c_void_p),
                ("slab_stride", ctypes.c_int64),
                ("slab_ptrs", ctypes.c_void_p),
                ("layout", q4moe_trellis_layout_t)]


class q4moe_options_t(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int64),
                ("gate_f32", ctypes.c_void_p),
                ("up_f32", ctypes.c_void_p),
                ("kernel", ctypes.c_int32),
                ("matvec_tile", ctypes.c_int32),
                ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_int64),
                ("tail", ctypes.c_int32),
                ("reserved1", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libq4moe.so (building it first if it is absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise Q4moeError(ERR_DEVICE, f"{path} is missing; run "
                                 "up_swiglu_gb300.build.build()")
            _build.build()
        lib = ctypes.CDLL(path)
        sig = {
            "q4moe_abi_version": (ctypes.c_int, []),
            "q4moe_last_error": (ctypes.c_char_p, []),
            "q4moe_canonical_layout": (ctypes.c_int, [_I64, _I64, _P]),
            "q4moe_canonical_layout_format": (ctypes.c_int,
                                              [_I64, _I64, _I32, _P]),
            "q4moe_validate_layout": (ctypes.c_int, [_P]),
            "q4moe_pack_slab": (ctypes.c_int, [_P, _P, _P, _P, _P, _P]),
            "q4moe_group_rows": (ctypes.c_int,
                                 [_P, _I64, _I32, _I32, _P, _P, _P, _P]),
            "q4moe_gate_up_swiglu": (ctypes.c_int,
                                     [_P, _P, _P, _P, _I64, _I64, _I64, _P,
                                      _P]),
            "q4moe_gate_up_swiglu_ex": (ctypes.c_int,
                                        [_P, _P, _P, _P, _I64, _I64, _I64,
                                         _P, _P, _P]),
            "q4moe_device_status": (ctypes.c_int,
                                    [_P, ctypes.POINTER(ctypes.c_uint32),
                                     ctypes.c_int]),
            "q4moe_debug_tail": (ctypes.c_int, [_P, _P, _I64, _P, _P]),
            "q4moe_debug_tail_mlx": (ctypes.c_int, [_P, _P, _I64, _P, _P]),
            "q4moe_debug_wait_timeout": (ctypes.c_int, [_I64, _P]),
            "q4moe_launch_count": (ctypes.c_int64, []),
            "q4moe_workspace_bytes": (ctypes.c_int64, [_I64, _I64]),
            "q4moe_gate_up_swiglu_noalloc": (ctypes.c_int,
                                             [_P, _P, _P, _P, _I64, _I64,
                                              _I64, _P, _P]),
            "q4moe_pack_slab_down": (ctypes.c_int, [_P, _P, _P, _P]),
            "q4moe_trellis_canonical_layout": (
                ctypes.c_int, [_I64, _I64, _I32, _I32, _I32, _I32, _P]),
            "q4moe_trellis_pack_slab": (ctypes.c_int,
                                        [_P, _P, _P, _P, _P, _P]),
            "q4moe_trellis_gate_up_swiglu": (
                ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _P, _P,
                               _P]),
            "q4moe_down_proj": (ctypes.c_int,
                                [_P, _P, _P, _I64, _I64, _I64, _P, _P, _P]),
            "q4moe_expert_mlp": (ctypes.c_int,
                                 [_P, _P, _P, _P, _I64, _I64, _I64, _P, _P,
                                  _P, _P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if lib.q4moe_abi_version() != ABI_VERSION:
            raise Q4moeError(ERR_DEVICE, "ABI version mismatch")
        _lib = lib
        return lib


def _check(rc: int) -> int:
    if rc != OK:
        raise Q4moeError(rc, load().q4moe_last_error().decode())
    return rc


def _ptr(t) -> int | None:
    """Device (or host) address of a tensor, array or raw integer."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):
        return t.ctypes.data
    raise TypeError(f"cannot take the address of {type(t)}")


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ------------------------------------------------------------- C functions --

def q4moe_abi_version() -> int:
    return load().q4moe_abi_version()


def q4moe_last_error() -> str:
    return load().q4moe_last_error().decode()


def q4moe_canonical_layout(H: int, I: int) -> q4moe_layout_t:
    L = q4moe_layout_t()
    _check(load().q4moe_canonical_layout(H, I, ctypes.byref(L)))
    return L


def q4moe_canonical_layout_format(H: int, I: int,
                                  fmt: int) -> q4moe_layout_t:
    L = q4moe_layout_t()
    _check(load().q4moe_canonical_layout_format(H, I, fmt, ctypes.byref(L)))
    return L


def q4moe_validate_layout(layout: q4moe_layout_t) -> None:
    _check(load().q4moe_validate_layout(ctypes.byref(layout)))


def q4moe_pack_slab(layout, gate_w, up_w, gate_s, up_s, slab_host) -> None:
    _check(load().q4moe_pack_slab(ctypes.byref(layout), _ptr(gate_w),
                                  _ptr(up_w), _ptr(gate_s), _ptr(up_s),
                                  _ptr(slab_host)))


def q4moe_pack_slab_down(layout, down_w, down_s, slab_host) -> None:
    _check(load().q4moe_pack_slab_down(ctypes.byref(layout), _ptr(down_w),
                                       _ptr(down_s), _ptr(slab_host)))


def q4moe_trellis_canonical_layout(H, I, block_size, window_bits, gate_bits,
                                   up_bits) -> q4moe_trellis_layout_t:
    L = q4moe_trellis_layout_t()
    _check(load().q4moe_trellis_canonical_layout(
        H, I, block_size, window_bits, gate_bits, up_bits, ctypes.byref(L)))
    return L


def q4moe_trellis_pack_slab(layout, gate_codes, up_codes, gate_scales,
                            up_scales, slab_host) -> None:
    _check(load().q4moe_trellis_pack_slab(
        ctypes.byref(layout), _ptr(gate_codes), _ptr(up_codes),
        _ptr(gate_scales), _ptr(up_scales), _ptr(slab_host)))


def q4moe_trellis_gate_up_swiglu(x, expert_slabs, row_offsets_per_expert,
                                 token_to_expert_map, M, H, I, out, opts=None,
                                 stream=None) -> None:
    _check(load().q4moe_trellis_gate_up_swiglu(
        _ptr(x), ctypes.byref(expert_slabs), _ptr(row_offsets_per_expert),
        _ptr(token_to_expert_map), M, H, I, _ptr(out),
        None if opts is None else ctypes.byref(opts), _stream(stream)))


def q4moe_group_rows(topk_ids, T, k, E, row_offsets, token_of_row,
                     row_of_pair, stream=None) -> None:
    _check(load().q4moe_group_rows(_ptr(topk_ids), T, k, E, _ptr(row_offsets),
                                   _ptr(token_of_row), _ptr(row_of_pair),
                                   _stream(stream)))


def q4moe_gate_up_swiglu(x, expert_slabs, row_offsets_per_expert,
                         token_to_expert_map, M, H, I, out,
                         stream=None) -> None:
    _check(load().q4moe_gate_up_swiglu(
        _ptr(x), ctypes.byref(expert_slabs), _ptr(row_offsets_per_expert),
        _ptr(token_to_expert_map), M, H, I, _ptr(out), _stream(stream)))


def q4moe_gate_up_swiglu_ex(x, expert_slabs, row_offsets_per_expert,
                            token_to_expert_map, M, H, I, out, opts=None,
                            stream=None) -> None:
    _check(load().q4moe_gate_up_swiglu_ex(
        _ptr(x), ctypes.byref(expert_slabs), _ptr(row_offsets_per_expert),
        _ptr(token_to_expert_map), M, H, I, _ptr(out),
        None if opts is None else ctypes.byref(opts), _stream(stream)))


def q4moe_gate_up_swiglu_noalloc(x, expert_slabs, row_offsets_per_expert,
                                 token_to_expert_map, M, H, I, out,
                                 stream=None) -> None:
    """The fused call without any device allocation: for callers that have
    no way to hand over scratch memory (see include/q4moe.h).  The scratch
    is a fixed array inside the library; M * H * 2 bytes must fit in
    NOALLOC_SCRATCH_BYTES."""
    _check(load().q4moe_gate_up_swiglu_noalloc(
        _ptr(x), ctypes.byref(expert_slabs), _ptr(row_offsets_per_expert),
        _ptr(token_to_expert_map), M, H, I, _ptr(out), _stream(stream)))


def q4moe_down_proj(mid, expert_slabs, row_offsets_per_expert, M, H, I, out,
                    opts=None, stream=None) -> None:
    _check(load().q4moe_down_proj(
        _ptr(mid), ctypes.byref(expert_slabs), _ptr(row_offsets_per_expert),
        M, H, I, _ptr(out), None if opts is None else ctypes.byref(opts),
        _stream(stream)))


def q4moe_expert_mlp(x, expert_slabs, row_offsets_per_expert,
                     token_to_expert_map, M, H, I, mid, out, opts=None,
                     stream=None) -> None:
    _check(load().q4moe_expert_mlp(
        _ptr(x), ctypes.byref(expert_slabs), _ptr(row_offsets_per_expert),
        _ptr(token_to_expert_map), M, H, I, _ptr(mid), _ptr(out),
        None if opts is None else ctypes.byref(opts), _stream(stream)))


def q4moe_device_status(stream=None, clear: bool = True) -> int:
    """Returns the status bits (0 when clean); never raises for set bits."""
    flags = ctypes.c_uint32(0)
    rc = load().q4moe_device_status(_stream(stream), ctypes.byref(flags),
                                    1 if clear else 0)
    if rc not in (OK, ERR_DEVICE_DATA):
        _check(rc)
    return int(flags.value)


def q4moe_workspace_bytes(M: int, H: int) -> int:
    n = int(load().q4moe_workspace_bytes(M, H))
    if n < 0:
        _check(n)
    return n


def q4moe_launch_count() -> int:
    return int(load().q4moe_launch_count())


def q4moe_debug_tail(gate_bf16, up_bf16, n, res, stream=None) -> None:
    _check(load().q4moe_debug_tail(_ptr(gate_bf16), _ptr(up_bf16), n,
                                   _ptr(res), _stream(stream)))


def q4moe_debug_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(load().q4moe_debug_wait_timeout(int(limit_ns), _stream(stream)))


def q4moe_debug_tail_mlx(gate_bf16, up_bf16, n, res, stream=None) -> None:
    _check(load().q4moe_debug_tail_mlx(_ptr(gate_bf16), _ptr(up_bf16), n,
                                       _ptr(res), _stream(stream)))


# ------------------------------------------------------- slab construction --

def make_slabs(num_experts: int, layout: q4moe_layout_t, base=None,
               slab_stride: int | None = None,
               slab_ptrs=None) -> q4moe_slabs_t:
    s = q4moe_slabs_t()
    s.num_experts = num_experts
    s.reserved0 = 0
    s.base = _ptr(base)
    s.slab_stride = layout.slab_bytes if slab_stride is None else slab_stride
    s.slab_ptrs = _ptr(slab_ptrs)
    s.layout = layout
    return s


def make_trellis_slabs(num_experts: int, layout: q4moe_trellis_layout_t,
                       base=None, slab_stride: int | None = None,
                       slab_ptrs=None) -> q4moe_trellis_slabs_t:
    s = q4moe_trellis_slabs_t()
    s.num_experts = num_experts
    s.reserved0 = 0
    s.base = _ptr(base)
    s.slab_stride = layout.slab_bytes if slab_stride is None else slab_stride
    s.slab_ptrs = _ptr(slab_ptrs)
    s.layout = layout
    return s


def pack_trellis_pool(layout: q4moe_trellis_layout_t, gate_codes, up_codes,
                      gate_scales, up_scales):
    """Host uint8 array [E, slab_bytes] of trellis slabs (codes uint32
    [E, I, words], f16 scale bit patterns [E, I])."""
    import numpy as np
    E = gate_codes.shape[0]
    pool = np.empty((E, layout.slab_bytes), dtype=np.uint8)
    for e in range(E):
        q4moe_trellis_pack_slab(layout, np.ascontiguousarray(gate_codes[e]),
                                np.ascontiguousarray(up_codes[e]),
                                np.ascontiguousarray(gate_scales[e]),
                                np.ascontiguousarray(up_scales[e]), pool[e])
    return pool


def pack_slab_pool(layout: q4moe_layout_t, gate_w, up_w, gate_s, up_s,
                   down_w=None, down_s=None):
    """Host uint8 array [E, slab_bytes] holding every expert's slab (numpy
    inputs [E, I, H/8] / [E, I], and optionally the down sections
    [E, H, I/8] / [E, H]); copy it to one 4096-aligned device allocation to
    use it."""
    import numpy as np
    E = gate_w.shape[0]
    pool = np.empty((E, layout.slab_bytes), dtype=np.uint8)
    for e in range(E):
        q4moe_pack_slab(layout, np.ascontiguousarray(gate_w[e]),
                        np.ascontiguousarray(up_w[e]),
                        np.ascontiguousarray(gate_s[e]),
                        np.ascontiguousarray(up_s[e]), pool[e])
        if down_w is not None:
            q4moe_pack_slab_down(layout, np.ascontiguousarray(down_w[e]),
                                 np.ascontiguousarray(down_s[e]), pool[e])
    return pool
