#!/usr/bin/env python3
"""Benchmark of the fused Q4 MoE expert gate/up + SwiGLU on one GB300.

One step = one pass of the whole path over one batch of synthetic input:
  * grouped workloads: token->expert grouping + the fused gate/up call
    (--op down: grouping + the down projection of synthetic intermediate
    activations; --op mlp: grouping + the whole expert MLP, gate/up then
    down);
  * the single-expert decode workload (H=4096, I=1536, one token): the call
    repeated 1000 times (the workload's own definition), each repeat on a
    different expert slab from a pool larger than 4x L2, captured once in a
    CUDA graph and replayed.
Inputs stay resident in HBM; every step streams its weights from HBM (the
weight pool of every workload is larger than L2).  Prints one JSON line for
the headline workload (by default the prefill, 160 experts, top-8, 4096
tokens, H=5120, I=1536: the largest one that fits one GPU) with a
"per_config" object holding the other workloads of the same operation and
format, timed in the same process (and the single-expert decode once more
with one slab reused, its weights L2-resident).

  python bench.py [--workload NAME] [--op gate_up|down|mlp] [--steps K]
                  [--warmup W] [--gpus N] [--no-per-config]
  python bench.py --impl reference ...   (the CPU oracle, timed alone)
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from up_swiglu_gb300 import synthetic as syn  # noqa: E402

METRIC = ("weight GB/s and TFLOP/s of Q4 MoE gate/up/SwiGLU; "
          "% of HBM / tensor roofline")
OP_METRIC = {
    "gate_up": METRIC,
    "down": ("weight GB/s and TFLOP/s of the Q4 MoE down projection; "
             "% of HBM / tensor roofline"),
    "mlp": ("weight GB/s and TFLOP/s of the Q4 MoE expert MLP (gate/up/"
            "SwiGLU, then down); % of HBM / tensor roofline"),
}


def swiglu_tail(fmt: str) -> str:
    """The tail a call in this format ends with under the default option
    (the pages' choice): MLX's compiled SwiGLU for trellis codes whose gate
    and up widths differ, page 52's otherwise."""
    if fmt.startswith("trellis"):
        kg, ku = fmt.split(":")[1].split(",")
        if kg != ku:
            return "mlx"
    return "page"


def op_metric(op: str, fmt: str) -> str:
    m = OP_METRIC[op]
    if fmt.startswith("trellis"):
        return m.replace("Q4", "trellis-coded")
    return m.replace("Q4", "Q8") if fmt == "q8" else m


OP_ENTRY = {"gate_up": "q4moe_gate_up_swiglu", "down": "q4moe_down_proj",
            "mlp": "q4moe_expert_mlp"}
DEFAULT_WORKLOAD = "moe160_top8_t4096_h5120_i1536"
# seconds of untimed steps, sampled for clocks, before the timed region
SUSTAIN_S = 1.0
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(syn.WORKLOADS))
    ap.add_argument("--format", default="q4",
                    choices=["q4", "q8", "trellis"],
                    help="weight format: packed nibbles (q4), signed bytes "
                         "(q8) or trellis codes (gate/up only)")
    ap.add_argument("--trellis-bits", default="4,4",
                    help="gate,up code widths of the trellis format")
    ap.add_argument("--op", default="gate_up",
                    choices=["gate_up", "down", "mlp"],
                    help="the gate/up call (default), the down projection, "
                         "or the whole expert MLP")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel", default="auto",
                    choices=["auto", "matvec", "gemm", "invariant"])
    ap.add_argument("--no-workspace", action="store_true",
                    help="call without the scratch workspace")
    ap.add_argument("--matvec-tile", type=int, default=0,
                    choices=[0, 16, 32, 64, 128],
                    help="unit height of the TMA matvec (0: per call)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time the headline workload only")
    ap.add_argument("--experts", type=int, default=0,
                    help="a reduced copy of the workload with this many "
                         "experts (profiling; 0: the workload's own)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="a reduced copy of the workload with this many "
                         "tokens (profiling; 0: the workload's own)")
    ap.add_argument("--sustain-seconds", type=float, default=SUSTAIN_S,
                    help="untimed steps sampled for clocks before the timed "
                         "region (0: none, e.g. under a profiler)")
    ap.add_argument("--l2-hot", action="store_true",
                    help="single-expert decode: every call on the same slab "
                         "(weights L2-resident)")
    return ap.parse_args(argv)


# ------------------------------------------------------------ workload math --

def workload_units(w: syn.Workload, topk: np.ndarray, E_pool: int,
                   op: str = "gate_up", fmt: str = "q4"):
    """Algorithmic work of one step: weight bytes (each touched expert's
    packed words + f32 scales, once per call), all bytes (+ activations read
    + outputs written) and flops.  gate/up: I*(H+8) weight bytes per expert,
    x read (2*H per token), out written (2*I per routed row), 4*H*I flops per
    routed row.  down: H*(I/2+4) weight bytes, mid read (2*I per row), out
    written (2*H per row), 2*H*I flops.  mlp: both, mid written and read
    back.  Q8: one byte per weight instead of half a byte."""
    per_byte = 1 if fmt == "q8" else 2           # weights per byte
    gu = w.I * (2 * w.H // per_byte + 8)
    if fmt.startswith("trellis"):                # trellis:kg,ku
        kg, ku = (int(v) for v in fmt.split(":")[1].split(","))
        gu = w.I * (w.H * (kg + ku) // 8 + 4)
    dn = w.H * (w.I // per_byte + 4)
    per_expert = {"gate_up": gu, "down": dn, "mlp": gu + dn}[op]
    rows = w.routed_rows
    act = {"gate_up": 2 * w.H * w.T + 2 * w.I * rows,
           "down": 2 * w.I * rows + 2 * w.H * rows,
           "mlp": 2 * w.H * w.T + 4 * w.I * rows + 2 * w.H * rows}[op]
    fl = {"gate_up": 4, "down": 2, "mlp": 6}[op] * w.H * w.I * rows
    if w.repeats > 1:
        calls = w.repeats
        touched = calls
        weight = calls * per_expert
        act *= calls
        fl *= calls
    else:
        touched = int(np.unique(topk).size)
        weight = touched * per_expert
    return dict(weight_bytes=weight, bytes=weight + act, flops=fl,
                touched_experts=touched)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(key: str):
    """DRAM bytes per call (the sum over the call's kernels) from the
    committed ncu summaries (profiles/ncu_traffic.txt), if every kernel's
    row was taken on its current source (sha256 prefix of the .cu file);
    else None."""
    import hashlib
    table = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    total, found = 0.0, False
    try:
        for line in open(table):
            parts = line.split()
            if len(parts) < 4 or line.startswith("#") or parts[0] != key:
                continue
            src = os.path.join(ROOT, "up_swiglu_gb300", "csrc", parts[1])
            sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
            if sha != parts[2]:
                return None                  # a kernel changed since
            total += float(parts[3])
            found = True
    except OSError:
        return None
    return total if found else None


# ---------------------------------------------------------------- clocks --

def device_smi_id(device_index: int) -> str:
    """The GPU's id for nvidia-smi --id: its UUID (unique under
    CUDA_VISIBLE_DEVICES, where the torch ordinal is not the physical
    index), else the ordinal."""
    try:
        import torch
        u = str(torch.cuda.get_device_properties(device_index).uuid)
        if u:
            return u if u.startswith(("GPU-", "MIG-")) else "GPU-" + u
    except Exception:           # noqa: BLE001 - any failure: the ordinal
        pass
    return str(device_index)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms.  mark()
    starts a new segment (e.g. the timed region after a sustain loop);
    summary() reports the whole run and each segment."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, device_index: int):
        self.dev = device_smi_id(device_index)
        self.proc = None
        self.file = None
        self.marks = []

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv",
                                                    delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}",
                 f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _rows(self):
        rows = []
        if self.file is None:
            return rows
        with open(self.file.name) as f:
            for line in f:
                if not line.endswith("\n"):
                    break                    # a row still being written
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        return rows

    def mark(self):
        """Start a new segment: the rows sampled from now on."""
        self.marks.append(len(self._rows()))

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    @staticmethod
    def _stats(rows):
        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        load = [r for r in rows if (num(r[9]) or 0.0) > 0.0]
        sm = [num(r[1]) for r in load if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for r in load:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "samples_under_load": len(load),
                "power_w_max": max(power) if power else None}

    def summary(self):
        """Clock statistics of the samples taken while the GPU was busy
        (utilization above 0), over the whole run, and per segment."""
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0, "segments": []}
        rows = self._rows()
        os.unlink(self.file.name)
        out = self._stats(rows)
        bounds = [0] + self.marks + [len(rows)]
        out["segments"] = [self._stats(rows[a:b])
                           for a, b in zip(bounds[:-1], bounds[1:])]
        return out


# ------------------------------------------------------------- GPU set-up --

class GpuWorkload:
    """Device-resident inputs for one workload and the step launcher."""

    def __init__(self, w: syn.Workload, kernel: str, device: int,
                 use_workspace: bool = True, matvec_tile: int = 0,
                 op: str = "gate_up", fmt: str = "q4",
                 l2_hot: bool = False):
        import torch
        from up_swiglu_gb300 import q4moe as q
        self.torch, self.q, self.w, self.op = torch, q, w, op
        self.kernel = {"auto": q.KERNEL_AUTO, "matvec": q.KERNEL_MATVEC,
                       "gemm": q.KERNEL_GEMM,
                       "invariant": q.KERNEL_BATCH_INVARIANT}[kernel]
        self.dev = torch.device("cuda", device)
        self.stream = torch.cuda.current_stream(self.dev)
        self.trellis = fmt.startswith("trellis")
        if self.trellis:
            kg, ku = (int(v) for v in fmt.split(":")[1].split(","))
            L = q.q4moe_trellis_canonical_layout(w.H, w.I, 256, 12, kg, ku)
        else:
            L = q.q4moe_canonical_layout_format(
                w.H, w.I, q.FORMAT_Q8 if fmt == "q8" else q.FORMAT_Q4)
        self.layout = L
        if w.repeats > 1 and l2_hot:
            pool_experts = 1                  # one slab, L2-resident
        elif w.repeats > 1:
            # distinct expert slabs, more than 4x L2 in total
            pool_experts = max(8, math.ceil(4 * L2_BYTES / L.slab_bytes) + 1)
            pool_experts = min(pool_experts, w.repeats)
        else:
            pool_experts = w.E
        self.pool_experts = pool_experts
        if self.trellis:
            g = syn.generate(w, experts=1)
            (g["gate_w"], g["up_w"], g["gate_s"],
             g["up_s"]) = syn.trellis_weights(w.seed, pool_experts, w.I, w.H,
                                              L.gate_bits, L.up_bits)
            host_pool = q.pack_trellis_pool(L, g["gate_w"], g["up_w"],
                                            g["gate_s"], g["up_s"])
        else:
            g = syn.generate(w, experts=pool_experts, fmt=fmt)
            if op != "gate_up":
                g.update(syn.generate_down(w, experts=pool_experts, fmt=fmt))
            host_pool = q.pack_slab_pool(L, g["gate_w"], g["up_w"],
                                         g["gate_s"], g["up_s"],
                                         g.get("down_w"), g.get("down_s"))
        self.host = g
        self.topk_host = g["topk"]
        nbytes = host_pool.size
        self._buf = torch.empty(nbytes + 4096, dtype=torch.uint8,
                                device=self.dev)
        off = (-self._buf.data_ptr()) % 4096
        self.pool = self._buf[off:off + nbytes]
        self.pool.copy_(torch.from_numpy(host_pool.reshape(-1)))
        del host_pool
        self.x = torch.from_numpy(g["x"].view(np.int16)).to(self.dev)
        self.topk = torch.from_numpy(g["topk"]).to(self.dev)
        self.M = w.routed_rows
        self.calls = w.repeats
        self.offs = torch.empty(w.E + 1, dtype=torch.int32, device=self.dev)
        self.tok = torch.empty(self.M, dtype=torch.int32, device=self.dev)
        self.rop = torch.empty(self.M, dtype=torch.int32, device=self.dev)
        self.out_cols = w.I if op == "gate_up" else w.H
        self.out = torch.empty((self.calls * self.M, self.out_cols),
                               dtype=torch.int16, device=self.dev)
        if op == "down":            # the down projection's input, resident
            self.mid = torch.from_numpy(g["mid"].view(np.int16)).to(self.dev)
        elif op == "mlp":           # the MLP's intermediate scratch
            self.mid = torch.empty((self.calls * self.M, w.I),
                                   dtype=torch.int16, device=self.dev)
        if w.repeats > 1:
            # single expert, single row: the grouping is the identity
            self.offs.copy_(torch.tensor([0, self.M], dtype=torch.int32))
            self.tok.zero_()
            mk = q.make_trellis_slabs if self.trellis else q.make_slabs
            self.slabs = [mk(1, L, base=self.pool.data_ptr() +
                             (r % pool_experts) * L.slab_bytes)
                          for r in range(self.calls)]
        else:
            mk = q.make_trellis_slabs if self.trellis else q.make_slabs
            self.slabs = [mk(w.E, L, base=self.pool)]
        self.opts = q.q4moe_options_t()
        self.opts.kernel = self.kernel
        self.opts.matvec_tile = matvec_tile
        self.opts_down = q.q4moe_options_t()
        self.opts_down.kernel = self.kernel
        self.opts_down.matvec_tile = matvec_tile
        if self.trellis:
            self.opts = q.q4moe_options_t()     # no kernel choice, no scratch
        elif use_workspace and op != "down":
            # scratch for the grouped activations the tensor-core GEMM reads
            nbytes = q.q4moe_workspace_bytes(self.M, w.H)
            self._ws = torch.empty(nbytes + 256, dtype=torch.uint8,
                                   device=self.dev)
            off = (-self._ws.data_ptr()) % 256
            self.opts.workspace = self._ws.data_ptr() + off
            self.opts.workspace_bytes = nbytes
        self.graph = None
        self.launches_per_step = None

    def _gate_up(self, r):
        """Call r of the step (one per repeat) through the library's entry
        point for the measured operation."""
        q, w = self.q, self.w
        out = self.out.data_ptr() + r * self.M * self.out_cols * 2
        if self.trellis:
            q.q4moe_trellis_gate_up_swiglu(self.x, self.slabs[r], self.offs,
                                           self.tok, self.M, w.H, w.I, out,
                                           self.opts, self.stream)
        elif self.op == "gate_up":
            q.q4moe_gate_up_swiglu_ex(self.x, self.slabs[r], self.offs,
                                      self.tok, self.M, w.H, w.I, out,
                                      self.opts, self.stream)
        elif self.op == "down":
            q.q4moe_down_proj(self.mid, self.slabs[r], self.offs, self.M,
                              w.H, w.I, out, self.opts_down, self.stream)
        else:
            mid = self.mid.data_ptr() + r * self.M * w.I * 2
            q.q4moe_expert_mlp(self.x, self.slabs[r], self.offs, self.tok,
                               self.M, w.H, w.I, mid, out, self.opts,
                               self.stream)

    def enqueue_step(self, ev=None):
        """Queue one step; ev = (start, mid) events bracket the grouping so
        the gate/up part can be timed on its own."""
        q = self.q
        if self.calls > 1:
            if self.graph is None:
                self._capture()
            if ev is not None:
                ev[0].record(self.stream)
                ev[1].record(self.stream)
            self.graph.replay()
            return
        if ev is not None:
            ev[0].record(self.stream)
        q.q4moe_group_rows(self.topk, self.w.T, self.w.topk, self.w.E,
                           self.offs, self.tok, self.rop, self.stream)
        if ev is not None:
            ev[1].record(self.stream)
        self._gate_up(0)

    def _capture(self):
        torch = self.torch
        for r in range(min(3, self.calls)):      # library set-up off-capture
            self._gate_up(r)
        torch.cuda.synchronize(self.dev)
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(self.dev)
        s.wait_stream(self.stream)
        n0 = self.q.q4moe_launch_count()
        with torch.cuda.graph(g, stream=s):
            saved = self.stream
            self.stream = s
            try:
                for r in range(self.calls):
                    self._gate_up(r)
            finally:
                self.stream = saved
        self.launches_per_step = self.q.q4moe_launch_count() - n0
        self.stream.wait_stream(s)
        self.graph = g


# ------------------------------------------------------------ CPU oracle ----

def oracle_sample(w: syn.Workload, g: dict, budget_s: float, nthreads=0,
                  op: str = "gate_up", fmt: str = "q4"):
    """Time the oracle on grouped rows (all outputs of each) until about
    budget_s seconds of work; returns (seconds per routed row, rows done,
    threads).  op down: the down projection of the rows of g["mid"]; op
    mlp: the rows' gate/up outputs, then their down outputs."""
    import oracle
    oracle.build()
    topk = g["topk"]
    E = g["gate_w"].shape[0]
    if w.repeats > 1:
        offs, tok = np.array([0, 1], np.int32), np.zeros(1, np.int32)
        Ew = 1
    else:
        offs, tok, _ = oracle.group_rows(topk, w.E)
        Ew = w.E
    M = int(offs[-1])
    rng = np.random.default_rng(0)
    rows_done, t_total = 0, 0.0
    order = rng.permutation(M) if M > 1 else np.zeros(1, np.int64)
    batch = max(1, min(M, 16))
    i = 0
    while t_total < budget_s:
        rows = order[i % M: i % M + batch] if M > 1 else order
        cols = np.tile(np.arange(w.I), rows.size)
        rr = np.repeat(rows, w.I)
        rh = np.repeat(rows, w.H)
        ch = np.tile(np.arange(w.H), rows.size)
        t0 = time.perf_counter()
        if fmt.startswith("trellis"):
            kg, ku = (int(v) for v in fmt.split(":")[1].split(","))
            r = oracle.trellis_gate_up_swiglu(
                g["x"], g["gate_w"][:Ew], g["up_w"][:Ew], g["gate_s"][:Ew],
                g["up_s"][:Ew], kg, ku, 12, 256, offs, tok, rr, cols,
                nthreads=nthreads, tail=swiglu_tail(fmt))
        elif op in ("gate_up", "mlp"):
            gu = oracle.q8_gate_up_swiglu if fmt == "q8" else \
                oracle.gate_up_swiglu_sampled
            r = gu(g["x"], g["gate_w"][:Ew], g["up_w"][:Ew], g["gate_s"][:Ew],
                   g["up_s"][:Ew], offs, tok, rr, cols, nthreads=nthreads)
        if op in ("down", "mlp"):
            if op == "mlp":
                mid = np.zeros((M, w.I), np.uint16)
                mid[rr, cols] = r["out"]
            else:
                mid = g["mid"][:M]
            dn = oracle.q8_down_proj if fmt == "q8" else \
                oracle.down_proj_sampled
            dn(mid, g["down_w"][:Ew], g["down_s"][:Ew], offs, rh, ch,
               nthreads=nthreads)
        t_total += time.perf_counter() - t0
        rows_done += rows.size
        i += batch
    del E
    return t_total / rows_done, rows_done, oracle.max_threads()


def cpu_value(w, units, sec_per_row):
    """Oracle throughput scaled to the whole step: weight GB/s."""
    rows_per_step = w.routed_rows * max(1, w.repeats)
    t_step = sec_per_row * rows_per_step
    return units["weight_bytes"] / t_step / 1e9, t_step


# --------------------------------------------------------------- replicas --

def max_over_ranks(ms: float, dist=None, device=None) -> float:
    """The slowest rank's time (every rank gets it); ms itself alone."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rates(units: dict, steps: int, world: int, total_ms: float):
    """Whole-job weight GB/s and TFLOP/s: every replica processes the same
    units per step, over the slowest replica's time."""
    sec = total_ms * 1e-3
    return (units["weight_bytes"] * steps * world / sec / 1e9,
            units["flops"] * steps * world / sec / 1e12)


# ------------------------------------------------------------------- main --

def run_reference(args, w, rank, world):
    """The reference arm: the CPU oracle as it stands, on the host cores,
    each step a bounded sample of the workload (rank 0 only)."""
    if rank != 0:
        return 0
    op = args.op
    fmt = args.format
    if fmt == "trellis":
        fmt = f"trellis:{args.trellis_bits}"
        kg, ku = (int(v) for v in args.trellis_bits.split(","))
        g = syn.generate(w, experts=1)
        (g["gate_w"], g["up_w"], g["gate_s"],
         g["up_s"]) = syn.trellis_weights(w.seed, w.E if w.repeats == 1
                                          else 1, w.I, w.H, kg, ku)
    else:
        g = syn.generate(w, experts=w.E if w.repeats == 1 else 1, fmt=fmt)
    if op != "gate_up":
        g.update(syn.generate_down(w, experts=w.E if w.repeats == 1 else 1,
                                   fmt=fmt))
    units = workload_units(w, g["topk"], w.E, op, fmt)
    per_step_budget = max(0.5, min(6.0, 150.0 / max(1, args.steps +
                                                    args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, g, per_step_budget / 4, op=op, fmt=fmt)
    times, rows = [], 0
    for _ in range(args.steps):
        spr, n, threads = oracle_sample(w, g, per_step_budget, op=op,
                                        fmt=fmt)
        times.append(spr)
        rows += n
    spr = statistics.mean(times)
    value, t_step = cpu_value(w, units, spr)
    line = {
        "impl": "reference", "metric": op_metric(op, fmt),
        "value": round(value, 4),
        "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded generator)",
        "config": {"workload": w.name, "op": op, "format": fmt, "E": w.E,
                   "H": w.H, "I": w.I, "tokens": w.T, "top_k": w.topk,
                   "routed_rows": w.routed_rows, "repeats": w.repeats,
                   "tail": swiglu_tail(fmt) if op != "down" else None},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s",
                         "cores": threads, "kind": "oracle",
                         "sample": f"{rows} routed rows x all their outputs "
                                   f"over {args.steps} steps, scaled to the "
                                   f"step's {w.routed_rows * w.repeats} rows"},
        "e2e": {"value": round(value, 4), "unit": "GB/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def l2_residency(gw):
    """How the step's weights sit against L2: more distinct slab bytes
    than L2 holds, or all of them resident after the first step."""
    total = gw.pool_experts * gw.layout.slab_bytes
    if total > L2_BYTES:
        return ("weights larger than L2 every step "
                f"({gw.pool_experts} distinct expert slabs, "
                f"{total / 2**20:.0f} MiB)")
    return (f"weights L2-resident ({gw.pool_experts} expert slab(s), "
            f"{total / 2**20:.1f} MiB, reused every step)")


def bracket_stride(steps: int) -> int:
    """Every how many timed steps the fused call is bracketed by events:
    8, or fewer so that at least 4 steps (all of them below 4) are."""
    return max(1, min(8, steps // 4))


def roofline_of(gw, w, units, op, fmt, per_launch_ms, peaks, peak_src,
                timed_s, l2_hot=False, kernel="auto", workspace=True):
    """Roofline of the fused call(s) of the operation: HBM for the decode
    kernels, the tensor core for the GEMM (burst peak unless the timed
    region lasts seconds).  The traffic of an L2-hot run has its own key
    (taken without cache flushes), and so have trellis widths other than
    4/4 and a forced kernel choice (other kernels, other bytes)."""
    rows_per_expert = (w.routed_rows if w.repeats > 1 else
                       w.routed_rows / units["touched_experts"])
    # (the trellis kernel decodes every weight once per 8 rows at any size:
    # its roofline is always the weight stream's)
    decode = rows_per_expert < 64 or fmt.startswith("trellis")
    traffic_key = w.name if op == "gate_up" else f"{w.name}:{op}"
    if fmt != "q4":
        traffic_key += ":" + (fmt if fmt.startswith("trellis:") and
                              fmt != "trellis:4,4" else fmt.split(":")[0])
    if kernel != "auto":
        traffic_key += ":" + kernel
    if not workspace and op != "down":
        traffic_key += ":no_workspace"
    if l2_hot:
        traffic_key += ":l2hot"
    if decode:
        bytes_per_launch = units["bytes"] / gw.calls
        achieved = bytes_per_launch / (per_launch_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        return {"bound": "hbm", "achieved": round(achieved, 2),
                "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": load_traffic(traffic_key),
                "kernel": ("q4moe_trellis_gate_up_swiglu (integer-bound "
                           "decode)" if gw.trellis
                           else f"{OP_ENTRY[op]} matvec"),
                "algorithmic_bytes_per_launch": int(bytes_per_launch),
                "peak_source": f"hbm_gbs of {peak_src}"}
    flops_per_launch = units["flops"] / gw.calls
    achieved = flops_per_launch / (per_launch_ms * 1e-3) / 1e12
    sustained = timed_s >= 2.0
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    peak = peaks[key]
    return {"bound": "tensor", "achieved": round(achieved, 2),
            "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4),
            "traffic": load_traffic(traffic_key),
            "kernel": f"{OP_ENTRY[op]} gemm (the call's launches: row copy "
                      "and tensor-core GEMM)",
            "algorithmic_flops_per_launch": int(flops_per_launch),
            "peak_source": f"{key} of {peak_src}"}


# Copies per step from which the end-to-end loop double-buffers (below, the
# streams' and events' host work costs more than the overlap gains: the
# small single expert measured 1.4 against 3.7 GB/s).
PIPELINE_MIN_BYTES = 256 * 1024


def e2e_time(gw, op, x_h, t_h, steps, copy_routing, pipeline=True):
    """Milliseconds per step end to end: every step copies its inputs from
    pinned host memory to the device and reads its outputs back.  A step of
    one call with enough bytes to copy double-buffers them (the copies of
    steps k + 1 and k - 1 run on two copy streams while step k computes); a
    graph of calls, whose buffers the graph fixes, and a small step copy in
    their stream's order.  Returns (ms, pipelined)."""
    import torch
    dev, stream = gw.dev, gw.stream
    in_name = "mid" if op == "down" else "x"
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if gw.graph is not None or not pipeline:
        o_h = torch.empty(gw.out.shape, dtype=torch.int16).pin_memory()
        x_dev = getattr(gw, in_name)
        e0.record(stream)
        for _ in range(steps):
            x_dev.copy_(x_h, non_blocking=True)
            if copy_routing:
                gw.topk.copy_(t_h, non_blocking=True)
            gw.enqueue_step()
            o_h.copy_(gw.out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / steps, False
    # two slots of the buffers the copies touch (inputs, routing, outputs);
    # the grouping, workspace and scratch are used by the compute stream only
    slots = [(getattr(gw, in_name), gw.topk, gw.out),
             (torch.empty_like(getattr(gw, in_name)),
              torch.empty_like(gw.topk), torch.empty_like(gw.out))]
    o_h = [torch.empty(gw.out.shape, dtype=torch.int16).pin_memory()
           for _ in range(2)]
    h2d_s = torch.cuda.Stream(dev)
    d2h_s = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_read = [torch.cuda.Event() for _ in range(2)]
    saved = slots[0]
    e0.record(stream)
    h2d_s.wait_event(e0)
    d2h_s.wait_event(e0)
    for k in range(steps):
        sl = k % 2
        x_d, t_d, out_d = slots[sl]
        with torch.cuda.stream(h2d_s):
            if k >= 2:                       # step k - 2 done with the slot
                h2d_s.wait_event(ev_done[sl])
            x_d.copy_(x_h, non_blocking=True)
            if copy_routing:
                t_d.copy_(t_h, non_blocking=True)
            ev_in[sl].record(h2d_s)
        stream.wait_event(ev_in[sl])
        if k >= 2:                           # step k - 2's outputs read
            stream.wait_event(ev_read[sl])
        setattr(gw, in_name, x_d)
        gw.topk, gw.out = t_d, out_d
        gw.enqueue_step()
        ev_done[sl].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(ev_done[sl])
            o_h[sl].copy_(out_d, non_blocking=True)
            ev_read[sl].record(d2h_s)
    stream.wait_stream(d2h_s)
    stream.wait_stream(h2d_s)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    setattr(gw, in_name, saved[0])
    gw.topk, gw.out = saved[1], saved[2]
    return e0.elapsed_time(e1) / steps, True


def measure(args, w, local, dist, world, rank, op, fmt, cpu_seconds,
            headline=False, l2_hot=False):
    """Set up one workload, time it (warm-up, then exactly args.steps steps
    between barriers and synchronisations), time it end to end with host
    buffers, and time the oracle on a bounded sample of it.  Returns the
    measured fields; the headline workload also samples clocks over an
    untimed sustain loop before its timed region."""
    import torch
    q = __import__("up_swiglu_gb300.q4moe", fromlist=["q4moe"])
    gw = GpuWorkload(w, args.kernel, local,
                     use_workspace=not args.no_workspace,
                     matvec_tile=args.matvec_tile, op=op, fmt=fmt,
                     l2_hot=l2_hot)
    units = workload_units(w, gw.topk_host, gw.pool_experts, op, fmt)
    dev = gw.dev
    stream = gw.stream

    # CPU baseline (host threads only, before the timed GPU work)
    cpu = None
    if rank == 0 and cpu_seconds > 0:
        spr, n, threads = oracle_sample(w, gw.host, cpu_seconds,
                                        op=op, fmt=fmt)
        v, _ = cpu_value(w, units, spr)
        cpu = {"value": round(v, 4), "unit": "GB/s", "cores": threads,
               "kind": "oracle",
               "sample": f"{n} routed rows x all their outputs "
                         f"(~{cpu_seconds:.0f} s), scaled to the step's "
                         f"{w.routed_rows * w.repeats} rows"}

    # warm-up
    for _ in range(max(args.warmup, 3)):
        gw.enqueue_step()
    torch.cuda.synchronize(dev)
    assert q.q4moe_device_status(stream, clear=True) == 0

    clk = ClockSampler(local) if headline else None
    if clk is not None:
        clk.__enter__()
    sustain = {"seconds": 0.0, "steps": 0}
    try:
        if clk is not None and args.sustain_seconds > 0:
            # untimed sustain loop (sampled)
            t0 = time.time()
            n_sus = 0
            while time.time() - t0 < args.sustain_seconds:
                for _ in range(8):
                    gw.enqueue_step()
                torch.cuda.synchronize(dev)
                n_sus += 8
            sustain = {"seconds": round(time.time() - t0, 3),
                       "steps": n_sus}
        if clk is not None:
            clk.mark()
        # timed region: K steps, barrier + synchronize on both sides.  The
        # fused call's own duration (the roofline's) is bracketed by events
        # on every stride-th step only: an event between two kernels keeps
        # the second from starting early (programmatic dependent launch),
        # and events on every step cost the grouped decode ~5 % of its step
        stride = bracket_stride(args.steps)
        ev = [(torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        ev_end = [torch.cuda.Event(enable_timing=True)
                  for _ in range(args.steps)]
        timed_calls = [k for k in range(args.steps)
                       if k % stride == stride - 1]
        n0 = q.q4moe_launch_count()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t_start = torch.cuda.Event(enable_timing=True)
        t_stop = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for k in range(args.steps):
            if k % stride == stride - 1:
                gw.enqueue_step(ev[k])
                ev_end[k].record(stream)
            else:
                gw.enqueue_step()
        t_stop.record(stream)
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        if clk is not None:
            clk.mark()
    finally:
        if clk is not None:
            clk.__exit__(None, None, None)
    launches = q.q4moe_launch_count() - n0
    if gw.graph is not None:
        launches = gw.launches_per_step * args.steps
    total_ms = t_start.elapsed_time(t_stop)
    call_ms = [ev[k][1].elapsed_time(ev_end[k]) for k in timed_calls]
    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_per_step = total_ms / args.steps
    value, tflops = job_rates(units, args.steps, world, total_ms)

    peaks, peak_src = load_peaks()
    per_launch_ms = statistics.mean(call_ms) / gw.calls
    roof = roofline_of(gw, w, units, op, fmt, per_launch_ms, peaks,
                       peak_src, total_ms * 1e-3, l2_hot=l2_hot,
                       kernel=args.kernel, workspace=not args.no_workspace)

    # end to end through the public API with host buffers: H2D of every
    # step's inputs (activations + routing) from pinned memory, D2H of its
    # outputs (the down projection's input is mid instead of x)
    x_src = gw.host["mid"] if op == "down" else gw.host["x"]
    x_h = torch.from_numpy(x_src.view(np.int16)).pin_memory()
    t_h = torch.from_numpy(gw.topk_host).pin_memory()
    h2d = x_h.numel() * 2 + (t_h.numel() * 4 if w.repeats == 1 else 0)
    d2h = gw.out.numel() * 2
    e2e_steps = max(3, min(args.steps, 10))
    e2e_ms, pipelined = e2e_time(gw, op, x_h, t_h, e2e_steps,
                                 copy_routing=w.repeats == 1,
                                 pipeline=h2d + d2h >= PIPELINE_MIN_BYTES)
    e2e_value = units["weight_bytes"] * world / (e2e_ms * 1e-3) / 1e9
    status = q.q4moe_device_status(stream, clear=True)
    res = {
        "gw": gw, "units": units, "ms_per_step": ms_per_step,
        "value": value, "tflops": tflops, "roofline": roof, "cpu": cpu,
        "e2e": {"value": round(e2e_value, 3), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "copies": ("overlapping the neighbouring steps' compute "
                           "(two buffer sets, two copy streams)"
                           if pipelined else "in the step's stream order")},
        "launches": int(launches), "status": status,
        "call_ms": statistics.mean(call_ms),
        "clocks": clk.summary() if clk is not None else None,
        "sustain": sustain,
        "l2": l2_residency(gw),
    }
    return res


def release(res):
    """Free a measured workload's device memory before the next one."""
    import torch
    res.pop("gw", None)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def per_config_entry(w, res, l2_hot=False):
    gw_pool = res["units"]["touched_experts"]
    return {
        "workload": w.name + (" (one slab reused: L2-resident weights)"
                              if l2_hot else ""),
        "routed_rows": w.routed_rows, "repeats": w.repeats,
        "touched_experts": gw_pool,
        "l2": res["l2"],
        "ms_per_step": round(res["ms_per_step"], 5),
        "value": round(res["value"], 3), "unit": "GB/s",
        "tflops": round(res["tflops"], 3),
        "roofline": res["roofline"],
        "cpu_baseline": res["cpu"],
        "e2e": res["e2e"],
        "gpu_launches": res["launches"],
        "device_status": res["status"],
    }


def main(argv=None):
    args = parse_args(argv)
    w = syn.WORKLOADS[args.workload]
    if args.experts or args.tokens:
        # a reduced copy for profiling: same shapes, routing and recipe
        import dataclasses
        E = args.experts or w.E
        T = args.tokens or w.T
        w = dataclasses.replace(w, name=f"{w.name}:E{E}:T{T}", E=E, T=T,
                                topk=min(w.topk, E))
        args.no_per_config = True
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, w, rank, world)

    import torch
    from up_swiglu_gb300 import q4moe as q
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    q.load()

    op, fmt = args.op, args.format
    if fmt == "trellis":
        if op != "gate_up":
            print(json.dumps({"error": "the trellis format has gate/up only"}))
            return 1
        fmt = f"trellis:{args.trellis_bits}"
    cpu_s = 0.0 if args.no_cpu_baseline else args.cpu_seconds

    # the other workloads of this operation and format first (each freed
    # before the next), then the headline one
    per_config = {}
    if not args.no_per_config:
        for name in sorted(syn.WORKLOADS,
                           key=lambda n: syn.WORKLOADS[n].routed_rows *
                           syn.WORKLOADS[n].E):
            if name == w.name:
                continue
            wc = syn.WORKLOADS[name]
            variants = [False] + ([True] if wc.repeats > 1 else [])
            for hot in variants:
                r = measure(args, wc, local, dist, world, rank, op, fmt,
                            0.0 if hot else max(1.0, cpu_s / 4),
                            l2_hot=hot)
                per_config[name + (":l2hot" if hot else "")] = \
                    per_config_entry(wc, r, hot)
                release(r)

    res = measure(args, w, local, dist, world, rank, op, fmt, cpu_s,
                  headline=True, l2_hot=args.l2_hot)
    gw, units = res["gw"], res["units"]
    clocks = res["clocks"]
    timed = clocks["segments"][1] if len(clocks["segments"]) > 1 else clocks
    sus = clocks["segments"][0] if len(clocks["segments"]) > 1 else None

    if rank == 0:
        line = {
            "metric": op_metric(op, fmt), "value": round(res["value"], 3),
            "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(res["ms_per_step"], 4),
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded generator; no dataset)",
            "config": {"workload": w.name, "op": op, "format": fmt,
                       "tail": swiglu_tail(fmt) if op != "down" else None,
                       "E": w.E, "H": w.H, "I": w.I,
                       "tokens": w.T, "top_k": w.topk,
                       "routed_rows": w.routed_rows, "repeats": w.repeats,
                       "touched_experts": units["touched_experts"],
                       "weight_bytes_per_step": units["weight_bytes"],
                       "flops_per_step": units["flops"],
                       "l2": res["l2"],
                       "kernel_choice": args.kernel,
                       "workspace": not args.no_workspace,
                       "matvec_tile": args.matvec_tile or "per call",
                       "parallelism": f"replicas x{world}" if world > 1
                       else "single GPU"},
            "tflops": round(res["tflops"], 3),
            "roofline": res["roofline"],
            "cpu_baseline": res["cpu"],
            "e2e": res["e2e"],
            "gpu_launches": res["launches"],
            # the timed region is too short for many samples (nvidia-smi
            # samples every 50 ms): the clock record covers the untimed
            # sustain loop of the same steps right before it as well
            "clocks": {"sm_mhz": clocks["sm_mhz"],
                       "sm_max_mhz": clocks["sm_max_mhz"],
                       "reasons": clocks["reasons"],
                       "samples": clocks["samples_under_load"],
                       "power_w_max": clocks["power_w_max"],
                       "window": "sustain loop of "
                                 f"{res['sustain']['seconds']} s + timed "
                                 "region",
                       "timed_region": {
                           "sm_mhz": timed["sm_mhz"],
                           "samples": timed["samples_under_load"],
                           "reasons": timed["reasons"]},
                       "sustain": None if sus is None else {
                           "sm_mhz": sus["sm_mhz"],
                           "samples": sus["samples_under_load"],
                           "reasons": sus["reasons"]}},
            "device_status": res["status"],
        }
        if per_config:
            line["per_config"] = per_config
        print(json.dumps(line), flush=True)
    release(res)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
