"""First launches of kernels never wait for code loading while another kernel holds SMs.

Under CUDA's lazy module loading a kernel's code is loaded at its first launch, and that
load can wait until the device is idle.  While the SM occupier spins on a host flag, such
a wait would last until the occupier's time limit.  gemm_create loads every kernel of the
library up front; this test runs in a fresh process with lazy loading forced on, starts
the occupier after one CLC launch and then makes first launches of other kernels, each
within the workspace the CLC launch sized (growing it synchronises the device, which
would wait for the occupier by design).  A regression is bounded: the occupier releases
its SMs after its 20 s limit."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, time
sys.path.insert(0, {root!r})
import torch
import workloads as wl
import blackwell_clc_dynamic_gb300 as clc
A = wl.make_matrix((128 * 40, 512), 211).cuda()
B = wl.make_matrix((512, 512), 212).cuda()
C = torch.empty((128 * 40, 512), device="cuda")
g = clc.Gemm(0)
s, so = torch.cuda.Stream(), torch.cuda.Stream()
g.run(A, B, C, stream=s)
s.synchronize()
g.occupy_start(24, limit_ns=20_000_000_000, stream=so)
g.occupy_wait_resident(10_000)
t0 = time.perf_counter()
g.run(A, B, C, sched="static", num_workers=64, stream=s)   # within the sized workspace
g.run(A, B, C, sched="nonpersistent", stream=s)
g.run(A, B, C, cluster=2, stream=s)
g.run(A, B, C, cluster=(2, 2, 1), stream=s)
s.synchronize()
dt = time.perf_counter() - t0
timed_out = g.occupy_stop()
torch.cuda.synchronize()
g.sync(s)
print("elapsed_s", dt, "occupier_timed_out", timed_out)
assert timed_out == 0 and dt < 5.0, dt
"""


def test_first_launches_do_not_wait_for_an_occupier():
    env = dict(os.environ, CUDA_MODULE_LOADING="LAZY")
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT)], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
