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
