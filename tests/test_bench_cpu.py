"""bench.py's host logic on CPU: the replica path (max of the ranks' times,
whole-job rates) over a world-size-2 gloo group, and the reference arm's
rank behaviour under a launcher."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], dist)
        units = {"weight_bytes": 1e9, "flops": 2e12}
        out.put((rank, ms, bench.job_rates(units, 10, world, ms)))
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_count_every_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [40.0, 50.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q))
             for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, (gbs, tflops) in res:
        assert ms == 50.0
        # 2 replicas x 10 steps x 1 GB in 50 ms; 2 x 10 x 2 TFLOP
        assert gbs == pytest.approx(2 * 10 * 1e9 / 0.05 / 1e9)
        assert tflops == pytest.approx(2 * 10 * 2e12 / 0.05 / 1e12)


def test_single_process_is_its_own_max():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5


def _reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world),
               LOCAL_RANK=str(rank))
    return subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl",
         "reference", "--workload", "expert1_h512_i256_m1", "--steps", "1",
         "--warmup", "0"], env=env, capture_output=True, text=True,
        timeout=300, cwd=ROOT)


def test_reference_arm_other_ranks_exit_quietly():
    r = _reference(1, 2)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    r = _reference(0, 2)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s",
                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_tail_reported_for_each_format():
    """The config's tail is the library's default choice: MLX's for
    trellis codes of different gate and up widths, page 52's otherwise."""
    import bench
    assert bench.swiglu_tail("q4") == "page"
    assert bench.swiglu_tail("q8") == "page"
    assert bench.swiglu_tail("trellis:4,4") == "page"
    assert bench.swiglu_tail("trellis:4,3") == "mlx"
    assert bench.swiglu_tail("trellis:2,4") == "mlx"


def test_clock_summary_keeps_busy_samples_and_segments(tmp_path):
    """Clock statistics come from the samples taken while the GPU was busy;
    mark() splits the run into a sustain segment and the timed region."""
    import bench
    rows = [
        # idx, sm, max, power, active, hw, hw_th, sw_th, sw_cap, util
        "0, 1995, 2070, 180.0, 0x0, Not Active, Not Active, Not Active, "
        "Not Active, 0",
        "0, 1800, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, "
        "Active, 100",
        "0, 1850, 2070, 1350.0, 0x0, Not Active, Not Active, Not Active, "
        "Not Active, 100",
        "0, 2000, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, "
        "Not Active, 97",
    ]
    clk = bench.ClockSampler.__new__(bench.ClockSampler)
    clk.proc = object()
    clk.file = open(tmp_path / "clk.csv", "w+")
    clk.marks = []
    clk.file.write("\n".join(rows[:3]) + "\n")
    clk.file.flush()
    clk.mark()
    clk.file.write(rows[3] + "\n" + "0, 17")   # last row still being written
    clk.file.flush()
    s = clk.summary()
    assert s["samples"] == 4 and s["samples_under_load"] == 3
    assert s["sm_mhz"] == 1850.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    sus, timed = s["segments"]
    assert sus["samples_under_load"] == 2 and sus["sm_mhz"] == 1825.0
    assert timed["samples_under_load"] == 1 and timed["sm_mhz"] == 2000.0
    assert timed["reasons"] == []


def test_gemm_roofline_takes_the_burst_peak_for_short_regions():
    """A tensor-bound line is compared with the burst bf16 peak unless the
    timed region lasts seconds; a decode line with the copy bandwidth."""
    import types
    import bench
    from up_swiglu_gb300 import synthetic as syn
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0,
             "bf16_tflops_sustained": 1700.0}
    gw = types.SimpleNamespace(calls=1, trellis=False)
    w = syn.WORKLOADS["moe160_top8_t4096_h5120_i1536"]
    units = {"touched_experts": 160, "bytes": 1.4e9, "flops": 1.0e12,
             "weight_bytes": 1.26e9}
    r = bench.roofline_of(gw, w, units, "gate_up", "q4", 1.0, peaks,
                          "measured", 0.1)
    assert r["bound"] == "tensor" and r["peak"] == 2000.0
    assert r["achieved"] == pytest.approx(1000.0)
    assert r["frac"] == pytest.approx(0.5)
    r = bench.roofline_of(gw, w, units, "gate_up", "q4", 1.0, peaks,
                          "measured", 5.0)
    assert r["peak"] == 1700.0
    w3 = syn.WORKLOADS["moe128_top8_t32_h5120_i1536"]
    units3 = {"touched_experts": 117, "bytes": 6.0e8, "flops": 8e9,
              "weight_bytes": 5.9e8}
    r = bench.roofline_of(gw, w3, units3, "gate_up", "q4", 0.2, peaks,
                          "measured", 0.1)
    assert r["bound"] == "hbm" and r["peak"] == 6000.0
    assert r["achieved"] == pytest.approx(3000.0)


def test_l2_residency_and_hot_traffic_key(monkeypatch):
    """The line says whether the step's distinct slab bytes exceed L2, and
    an L2-hot run looks its DRAM traffic up under its own key."""
    import types
    import bench
    from up_swiglu_gb300 import synthetic as syn
    small = types.SimpleNamespace(pool_experts=1,
                                  layout=types.SimpleNamespace(
                                      slab_bytes=133_120))
    big = types.SimpleNamespace(pool_experts=83,
                                layout=types.SimpleNamespace(
                                    slab_bytes=6_316_032))
    assert bench.l2_residency(small).startswith("weights L2-resident")
    assert bench.l2_residency(big).startswith("weights larger than L2")
    keys = []
    monkeypatch.setattr(bench, "load_traffic",
                        lambda k: keys.append(k) or None)
    gw = types.SimpleNamespace(calls=1000, trellis=False)
    w = syn.WORKLOADS["expert1_h4096_i1536_m1_x1000"]
    units = {"touched_experts": 1000, "bytes": 6.3e9, "flops": 2.5e10,
             "weight_bytes": 6.3e9}
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0,
             "bf16_tflops_sustained": 1700.0}
    bench.roofline_of(gw, w, units, "gate_up", "q4", 0.005, peaks,
                      "measured", 0.1)
    bench.roofline_of(gw, w, units, "gate_up", "q4", 0.005, peaks,
                      "measured", 0.1, l2_hot=True)
    assert keys == [w.name, w.name + ":l2hot"]


def test_traffic_key_names_width_and_forced_kernel(monkeypatch):
    """Traffic rows are per kernel set: trellis widths other than 4/4 and a
    forced kernel choice look up keys of their own."""
    import types
    import bench
    from up_swiglu_gb300 import synthetic as syn
    keys = []
    monkeypatch.setattr(bench, "load_traffic",
                        lambda k: keys.append(k) or None)
    gw = types.SimpleNamespace(calls=1, trellis=False)
    w = syn.WORKLOADS["moe128_top8_t32_h5120_i1536"]
    units = {"touched_experts": 117, "bytes": 6.0e8, "flops": 8e9,
             "weight_bytes": 5.9e8}
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0,
             "bf16_tflops_sustained": 1700.0}
    for fmt, kernel in [("trellis:4,4", "auto"), ("trellis:4,3", "auto"),
                        ("q8", "auto"), ("q4", "matvec")]:
        bench.roofline_of(gw, w, units, "gate_up", fmt, 0.2, peaks,
                          "measured", 0.1, kernel=kernel)
    bench.roofline_of(gw, w, units, "gate_up", "q4", 0.2, peaks, "measured",
                      0.1, workspace=False)
    assert keys == [w.name + ":trellis", w.name + ":trellis:4,3",
                    w.name + ":q8", w.name + ":matvec",
                    w.name + ":no_workspace"]


def test_bracket_stride_samples_at_least_four_steps():
    """The fused call is timed on every stride-th step: 8 for long runs,
    at least 4 samples when there are 4 steps or more, every step below."""
    import bench
    assert bench.bracket_stride(100) == 8
    assert bench.bracket_stride(20) == 5
    assert bench.bracket_stride(3) == 1 and bench.bracket_stride(1) == 1
    for k in range(1, 200):
        s = bench.bracket_stride(k)
        n = sum(1 for i in range(k) if i % s == s - 1)
        assert n >= min(k, 4)
