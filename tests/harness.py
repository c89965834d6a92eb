"""Host/GPU plumbing shared by the GPU tests: build a problem from the seeded
generator, upload it, and call the library through its C ABI binding.
PyTorch only allocates device memory and provides the stream."""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from up_swiglu_gb300 import q4moe as q
from up_swiglu_gb300 import synthetic as syn


@dataclass
class Problem:
    x: np.ndarray         # bf16 bits [T, H]
    gate_w: np.ndarray    # uint32 [E, I, H/8]
    up_w: np.ndarray
    gate_s: np.ndarray    # f32 [E, I]
    up_s: np.ndarray
    topk: np.ndarray      # int32 [T, k]
    down_w: np.ndarray = None   # uint32 [E, H, I/8] (optional)
    down_s: np.ndarray = None   # f32 [E, H]

    @property
    def E(self):
        return self.gate_w.shape[0]

    @property
    def I(self):
        return self.gate_w.shape[1]

    @property
    def H(self):
        return self.x.shape[1]

    @property
    def T(self):
        return self.x.shape[0]

    @property
    def k(self):
        return self.topk.shape[1]


def random_problem(seed, E, I, H, T, k, routing="uniform", x_std=1.0):
    x = syn.normal_x(seed, T, H, x_std)
    gw, uw, gs, us = syn.weights(seed, E, I, H)
    if routing == "uniform":
        topk = syn.route_uniform(seed, T, k, E)
    elif routing == "zipf":
        topk = syn.route_zipf(seed, T, k, E, 1.1)
    else:
        raise ValueError(routing)
    return Problem(x, gw, uw, gs, us, topk)


def exact_problem(seed, E, I, H, T, k):
    x, gw, uw, gs, us = syn.exact_integer_case(seed, T, H, E, I)
    return Problem(x, gw, uw, gs, us, syn.route_uniform(seed, T, k, E))


def problem_with_counts(seed, counts, I, H, exact=False):
    """One token per routed row, expert e getting counts[e] rows."""
    E = len(counts)
    T = int(sum(counts))
    ids = np.concatenate([np.full(c, e, np.int32)
                          for e, c in enumerate(counts)])
    ids = ids[np.random.default_rng(seed).permutation(T)] if T else ids
    if exact:
        x, gw, uw, gs, us = syn.exact_integer_case(seed, max(T, 1), H, E, I)
        x = x[:T]
    else:
        x = syn.normal_x(seed, T, H)
        gw, uw, gs, us = syn.weights(seed, E, I, H)
    return Problem(x, gw, uw, gs, us, ids.reshape(T, 1))


def aligned_device_buffer(nbytes, align=q.SLAB_ALIGNMENT):
    import torch
    buf = torch.empty(nbytes + align, dtype=torch.uint8, device="cuda")
    off = (-buf.data_ptr()) % align
    return buf, buf[off:off + nbytes]


@dataclass
class DeviceProblem:
    p: Problem
    layout: object
    slabs: object
    keep: list = field(default_factory=list)
    x: object = None
    topk: object = None


def upload(p: Problem, layout=None, stride_pad=0, ptr_table=False,
           x_offset=0):
    """Pack the experts into slabs (canonical layout unless given), copy them
    into one 4096-aligned device pool, and upload x and the routing (x_offset
    bf16 elements past a 256-byte boundary)."""
    import torch
    L = layout or q.q4moe_canonical_layout(p.H, p.I)
    host = q.pack_slab_pool(L, p.gate_w, p.up_w, p.gate_s, p.up_s,
                            p.down_w, p.down_s)
    stride = L.slab_bytes + stride_pad
    keep = []
    buf, pool = aligned_device_buffer(p.E * stride)
    keep.append(buf)
    if stride == L.slab_bytes:
        pool.copy_(torch.from_numpy(host.reshape(-1)))
    else:
        for e in range(p.E):
            pool[e * stride:e * stride + L.slab_bytes].copy_(
                torch.from_numpy(host[e]))
    if ptr_table:
        # slots in a shuffled order: expert e lives in slot perm[e]
        perm = np.random.default_rng(p.E).permutation(p.E)
        buf2, pool2 = aligned_device_buffer(p.E * stride)
        keep.append(buf2)
        for e in range(p.E):
            pool2[perm[e] * stride:perm[e] * stride + L.slab_bytes].copy_(
                pool[e * stride:e * stride + L.slab_bytes])
        ptrs = torch.tensor([pool2.data_ptr() + int(perm[e]) * stride
                             for e in range(p.E)], dtype=torch.int64,
                            device="cuda")
        keep.append(ptrs)
        slabs = q.make_slabs(p.E, L, slab_ptrs=ptrs)
    else:
        slabs = q.make_slabs(p.E, L, base=pool, slab_stride=stride)
    d = DeviceProblem(p, L, slabs, keep)
    xh = torch.from_numpy(np.ascontiguousarray(p.x).view(np.int16))
    if x_offset:
        xbuf, xv = aligned_device_buffer(xh.numel() * 2 + 2 * x_offset, 256)
        keep.append(xbuf)
        d.x = xv.view(torch.int16)[x_offset:x_offset + xh.numel()] \
            .view(xh.shape)
        d.x.copy_(xh)
    else:
        d.x = xh.cuda()
    d.topk = torch.from_numpy(np.ascontiguousarray(p.topk)).cuda()
    return d


def group(d: DeviceProblem, stream=None):
    import torch
    n = d.p.T * d.p.k
    offs = torch.empty(d.p.E + 1, dtype=torch.int32, device="cuda")
    tok = torch.empty(max(n, 1), dtype=torch.int32, device="cuda")
    rop = torch.empty(max(n, 1), dtype=torch.int32, device="cuda")
    q.q4moe_group_rows(d.topk, d.p.T, d.p.k, d.p.E, offs, tok, rop, stream)
    return offs, tok[:n], rop[:n]


def gate_up(d: DeviceProblem, offs, tok, kernel=q.KERNEL_AUTO, debug=True,
            stream=None, out=None, workspace=False, matvec_tile=0):
    """Run the fused call; returns numpy out bits [M, I] (+ gate32/up32).
    workspace=True hands the call a scratch buffer (grouped activations
    for the tensor-core GEMM); matvec_tile fixes the TMA matvec's unit
    height."""
    import torch
    M = int(tok.shape[0])
    I = d.p.I
    if out is None:
        out = torch.full((max(M, 1), I), -1, dtype=torch.int16,
                         device="cuda")
    res = {}
    if debug or kernel != q.KERNEL_AUTO or workspace or matvec_tile:
        g32 = torch.full((max(M, 1), I), float("nan"), device="cuda") \
            if debug else None
        u32 = torch.full((max(M, 1), I), float("nan"), device="cuda") \
            if debug else None
        o = q.q4moe_options_t()
        o.num_tokens = d.p.T
        o.gate_f32 = None if g32 is None else g32.data_ptr()
        o.up_f32 = None if u32 is None else u32.data_ptr()
        o.kernel = kernel
        o.matvec_tile = matvec_tile
        if workspace:
            nbytes = q.q4moe_workspace_bytes(M, d.p.H)
            wbuf, ws = aligned_device_buffer(max(nbytes, 256), 256)
            ws.fill_(0xFF)                      # stale contents must not matter
            d.keep.append(wbuf)
            o.workspace = ws.data_ptr()
            o.workspace_bytes = nbytes
        q.q4moe_gate_up_swiglu_ex(d.x, d.slabs, offs, tok, M, d.p.H, I, out,
                                  o, stream)
        if debug:
            res["gate32"] = g32[:M].cpu().numpy()
            res["up32"] = u32[:M].cpu().numpy()
    else:
        q.q4moe_gate_up_swiglu(d.x, d.slabs, offs, tok, M, d.p.H, I, out,
                               stream)
    torch.cuda.synchronize()
    res["out"] = out[:M].cpu().numpy().view(np.uint16)
    return res


def element_scales(p: Problem, offs: np.ndarray):
    """gate/up scale of every output element [M, I] (grouped order)."""
    M = int(offs[-1])
    e_of_row = np.repeat(np.arange(p.E), np.diff(offs))
    assert e_of_row.shape[0] == M
    return p.gate_s[e_of_row], p.up_s[e_of_row]


def with_down(p: Problem, seed, exact=False) -> Problem:
    """p with down sections drawn from the seeded generator (power-of-two
    scales when exact)."""
    dw, ds = syn.down_weights(seed, p.E, p.H, p.I)
    if exact:
        _, dw, ds = syn.exact_down_case(seed, 1, p.I, p.E, p.H)
    p.down_w, p.down_s = dw, ds
    return p


def down_only_problem(seed, counts, K, N, exact=False, mid_std=0.1):
    """A down projection on its own: expert e gets counts[e] grouped rows of
    mid (bf16 [M, K]); N output rows.  Returns (Problem, mid bits,
    row_offsets).  The gate/up sections are filler (never read)."""
    E, M = len(counts), int(sum(counts))
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    if exact:
        mid, dw, ds = syn.exact_down_case(seed, max(M, 1), K, E, N)
        mid = mid[:M]
    else:
        mid = syn.normal_x(seed, max(M, 1), K, std=mid_std,
                           stream=syn.S_EXACT_MID)[:M]
        dw, ds = syn.down_weights(seed, E, N, K)
    gw = np.zeros((E, K, N // 8), np.uint32)
    gs = np.zeros((E, K), np.float32)
    p = Problem(np.zeros((1, N), np.uint16), gw, gw, gs, gs,
                np.zeros((1, 1), np.int32), dw, ds)
    return p, mid, offs


def down(d: DeviceProblem, offs, mid, kernel=q.KERNEL_AUTO, debug=True,
         matvec_tile=0, stream=None, mid_offset=0):
    """Run q4moe_down_proj on mid (numpy bits [M, I] or a device tensor);
    returns numpy out bits [M, H] (+ out32)."""
    import torch
    H, I = d.p.H, d.p.I
    if isinstance(mid, np.ndarray):
        M = mid.shape[0]
        mh = torch.from_numpy(np.ascontiguousarray(mid).view(np.int16))
        mbuf, md = aligned_device_buffer(max(mh.numel(), 1) * 2 +
                                         2 * mid_offset, 256)
        d.keep.append(mbuf)
        md = md.view(torch.int16)[mid_offset:mid_offset + mh.numel()]
        md.copy_(mh.reshape(-1))
    else:
        md = mid
        M = mid.shape[0] if mid.dim() == 2 else mid.numel() // I
    offs_d = offs if not isinstance(offs, np.ndarray) else \
        torch.from_numpy(offs).cuda()
    out = torch.full((max(M, 1), H), -1, dtype=torch.int16, device="cuda")
    o = q.q4moe_options_t()
    o.kernel = kernel
    o.matvec_tile = matvec_tile
    o32 = None
    if debug:
        o32 = torch.full((max(M, 1), H), float("nan"), device="cuda")
        o.gate_f32 = o32.data_ptr()
    q.q4moe_down_proj(md, d.slabs, offs_d, M, H, I, out, o, stream)
    torch.cuda.synchronize()
    res = {"out": out[:M].cpu().numpy().view(np.uint16)}
    if debug:
        res["out32"] = o32[:M].cpu().numpy()
    return res


def expert_mlp(d: DeviceProblem, offs, tok, kernel=q.KERNEL_AUTO,
               debug=True, workspace=False, matvec_tile=0, stream=None):
    """Run q4moe_expert_mlp; returns numpy mid bits [M, I], out bits [M, H]
    (+ gate32/up32 of the gate/up stage)."""
    import torch
    M = int(tok.shape[0])
    H, I = d.p.H, d.p.I
    mid = torch.full((max(M, 1), I), -1, dtype=torch.int16, device="cuda")
    out = torch.full((max(M, 1), H), -1, dtype=torch.int16, device="cuda")
    o = q.q4moe_options_t()
    o.num_tokens = d.p.T
    o.kernel = kernel
    o.matvec_tile = matvec_tile
    g32 = u32 = None
    if debug:
        g32 = torch.full((max(M, 1), I), float("nan"), device="cuda")
        u32 = torch.full((max(M, 1), I), float("nan"), device="cuda")
        o.gate_f32, o.up_f32 = g32.data_ptr(), u32.data_ptr()
    if workspace:
        nbytes = q.q4moe_workspace_bytes(M, H)
        wbuf, ws = aligned_device_buffer(max(nbytes, 256), 256)
        ws.fill_(0xFF)
        d.keep.append(wbuf)
        o.workspace = ws.data_ptr()
        o.workspace_bytes = nbytes
    q.q4moe_expert_mlp(d.x, d.slabs, offs, tok, M, H, I, mid, out, o, stream)
    torch.cuda.synchronize()
    res = {"mid": mid[:M].cpu().numpy().view(np.uint16),
           "out": out[:M].cpu().numpy().view(np.uint16)}
    if debug:
        res["gate32"] = g32[:M].cpu().numpy()
        res["up32"] = u32[:M].cpu().numpy()
    return res


def down_scales(p: Problem, offs: np.ndarray):
    """down scale of every output element [M, H] (grouped order)."""
    e_of_row = np.repeat(np.arange(p.E), np.diff(offs))
    return p.down_s[e_of_row]


def q8_layout(p: Problem):
    return q.q4moe_canonical_layout_format(p.H, p.I, q.FORMAT_Q8)


def q8_problem(seed, E, I, H, T, k, exact=False, routing="uniform",
               with_down=True):
    """A Q8 problem (int8 weights) with its down sections."""
    if exact:
        x, gw, uw, gs, us = syn.exact_q8_case(seed, T, H, E, I)
    else:
        x = syn.normal_x(seed, T, H)
        gw, uw, gs, us = syn.q8_weights(seed, E, I, H)
    topk = syn.route_uniform(seed, T, k, E) if routing == "uniform" else \
        syn.route_zipf(seed, T, k, E, 1.1)
    p = Problem(x, gw, uw, gs, us, topk)
    if with_down:
        p.down_w, p.down_s = syn.q8_down_weights(seed, E, H, I)
        if exact:
            ks = (syn.u64(seed, syn.S_EXACT_DS, E * H) % np.uint64(6)) \
                .astype(np.int64) + 8
            p.down_s = np.ldexp(np.float32(1.0), -ks).astype(
                np.float32).reshape(E, H)
    return p


def q8_counts_problem(seed, counts, I, H, exact=False):
    """Q8, one token per routed row, expert e getting counts[e] rows."""
    E = len(counts)
    T = int(sum(counts))
    ids = np.concatenate([np.full(c, e, np.int32)
                          for e, c in enumerate(counts)])
    ids = ids[np.random.default_rng(seed).permutation(T)] if T else ids
    p = q8_problem(seed, E, I, H, max(T, 1), 1, exact=exact)
    p.x = p.x[:T]
    p.topk = ids.reshape(T, 1)
    return p


def q8_down_only_problem(seed, counts, K, N, exact=False, mid_std=0.1):
    """Q8 down projection on its own (see down_only_problem)."""
    E, M = len(counts), int(sum(counts))
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    if exact:
        mi = (syn.u64(seed, syn.S_EXACT_MID, max(M, 1) * K) %
              np.uint64(17)).astype(np.int64) - 8
        mid = syn.f32_to_bf16_bits(mi.astype(np.float32)).reshape(-1, K)[:M]
    else:
        mid = syn.normal_x(seed, max(M, 1), K, std=mid_std,
                           stream=syn.S_MID)[:M]
    dw, ds = syn.q8_down_weights(seed, E, N, K)
    if exact:
        ks = (syn.u64(seed, syn.S_EXACT_DS, E * N) % np.uint64(6)).astype(
            np.int64) + 8
        ds = np.ldexp(np.float32(1.0), -ks).astype(np.float32).reshape(E, N)
    gw = np.zeros((E, K, N), np.int8)
    gs = np.zeros((E, K), np.float32)
    p = Problem(np.zeros((1, N), np.uint16), gw, gw, gs, gs,
                np.zeros((1, 1), np.int32), dw, ds)
    return p, mid, offs
