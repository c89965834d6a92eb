"""The boundary's promises on a GPU: the bounded on-chip waits give up and
report instead of hanging, and no call needs set-up work of its own (the
first call of a fresh process can be captured in a CUDA graph)."""
from __future__ import annotations

import os
import subprocess
import sys

import numpy as np
import pytest

import harness as hz
from up_swiglu_gb300 import q4moe as q

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    q.load()
    q.q4moe_device_status(clear=True)
    yield


def test_bounded_wait_runs_out_and_reports():
    """An mbarrier nothing arrives on, waited on as the kernels wait (the
    try_wait loop and the MMA issuer's spin) with a 1 ms limit: the kernel
    returns, the status word carries Q4MOE_DEV_WAIT_TIMEOUT, and the next
    call works as before."""
    import time
    import torch
    p = hz.problem_with_counts(3, [5, 0, 9], 256, 512, exact=True)
    d = hz.upload(p)
    offs, tok, _ = hz.group(d)
    before = hz.gate_up(d, offs, tok)["out"]
    assert q.q4moe_device_status(clear=True) == 0
    t0 = time.time()
    q.q4moe_debug_wait_timeout(1000000)
    torch.cuda.synchronize()
    assert time.time() - t0 < 5.0
    flags = q.q4moe_device_status(clear=True)
    assert flags == q.DEV_WAIT_TIMEOUT
    after = hz.gate_up(d, offs, tok)["out"]
    assert np.array_equal(before, after)
    assert q.q4moe_device_status(clear=True) == 0


_CAPTURE_FIRST_CALL = r"""
import sys
sys.path.insert(0, {root!r})
sys.path.insert(0, {tests!r})
import numpy as np, torch
import harness as hz
from up_swiglu_gb300 import q4moe as q
q.load()
p = hz.problem_with_counts(11, [7, 3, 12], 256, 512, exact=True)
d = hz.upload(p)
offs = torch.tensor(np.concatenate([[0], np.cumsum([7, 3, 12])]),
                    dtype=torch.int32, device="cuda")
order = np.argsort(p.topk.ravel(), kind="stable").astype(np.int32)
tok = torch.from_numpy(order).cuda()
out = torch.full((22, 256), -1, dtype=torch.int16, device="cuda")
torch.cuda.synchronize()
g = torch.cuda.CUDAGraph()
s = torch.cuda.Stream()
with torch.cuda.stream(s):
    with torch.cuda.graph(g, stream=s):
        # the process's first call of the library on this device
        q.q4moe_gate_up_swiglu(d.x, d.slabs, offs, tok, 22, 512, 256, out,
                               s.cuda_stream)
g.replay()
torch.cuda.synchronize()
want = torch.full((22, 256), -1, dtype=torch.int16, device="cuda")
q.q4moe_gate_up_swiglu(d.x, d.slabs, offs, tok, 22, 512, 256, want)
torch.cuda.synchronize()
assert torch.equal(out, want), "captured first call differs"
assert q.q4moe_device_status(clear=True) == 0
print("first call captured")
"""


def test_first_call_of_a_process_can_be_captured():
    """A fresh process whose very first library call is made during stream
    capture: the call records its kernels like any other (nothing is
    launched or waited on for set-up), and the replayed graph gives the
    same bits as a plain call."""
    code = _CAPTURE_FIRST_CALL.format(root=ROOT,
                                      tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True,
                       text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "first call captured" in r.stdout
