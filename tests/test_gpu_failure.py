"""Failure detection without a GPU fault: every device-side wait is bounded, and a wait
that runs out is reported through the device error word while the context stays usable.

The hold_scheduler hook makes the CLC scheduler issue and signal nothing (a response
that nothing ever delivers).  Every worker still computes its own launch's tile, then
its response waits run out after timeout_ns; nothing is in flight by then (the tile
finished microseconds earlier), so the CTA unwinds, frees its tensor memory and exits.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_helpers import TILE_256, assert_close, check_log, cluster_dims

pytestmark = pytest.mark.gpu

WAIT_CLC_FULL = 5


@pytest.mark.parametrize("cl,mc", [(1, 0), (2, 0), (4, 0), ((2, 2, 1), 0)], ids=["c1", "c2pair", "c4mc", "c2x2"])
def test_response_wait_times_out_and_is_reported(cl, mc):
    import blackwell_clc_dynamic_gb300 as m
    ncta, rm, rn = cluster_dims(cl)
    M, N, K = 128 * rm * 6, 512 * rn, 256
    A = wl.make_matrix((M, K), 101)
    B = wl.make_matrix((K, N), 102)
    with m.Gemm(0, timeout_ns=50_000_000, hold_scheduler=True, cluster_b_multicast=mc) as g:
        C = torch.full((M, N), float("nan"), device="cuda")
        g.run(A.cuda(), B.cuda(), C, tile=TILE_256, cluster=cl, sched="clc")
        torch.cuda.synchronize()
        bits, site, block = g.device_error()
        assert bits == 1 and site == WAIT_CLC_FULL
        with pytest.raises(m.GemmError) as ei:
            g.sync()
        assert ei.value.code == m.GEMM_ERR_TIMEOUT
        # nothing was stolen: every launch computed its own tile, exactly once
        assert_close(C.cpu().numpy(), oracle.gemm(A, B))
        owner_lin, first = check_log(g, "nonpersistent", [6], 2, ncta, rn=rn)
        # the error word was cleared by gemm_sync, and the context still works
        g.set_opts(hold_scheduler=0, timeout_ns=0)
        C2 = torch.full((M, N), float("nan"), device="cuda")
        g.run(A.cuda(), B.cuda(), C2, tile=TILE_256, cluster=cl, sched="clc")
        g.sync()
        assert g.device_error() == (0, 0, 0)
        assert_close(C2.cpu().numpy(), oracle.gemm(A, B))


def test_higher_priority_kernels_stop_fetching_but_keep_coverage():
    """A cancel may fail because the hardware wants to schedule a higher-priority kernel
    ("CUTLASS CLC dynamic persistent kernel", section "Cluster granularity and exit after
    failure").  A CLC GEMM runs on a low-priority stream; right after it, an occupier that
    cannot share an SM with it (large shared-memory footprint) is launched on a
    higher-priority stream.  Workers whose cancel fails stop and give their SM up; the
    launches nobody took run later.  Every tile is still computed exactly once."""
    import blackwell_clc_dynamic_gb300 as m
    M, N, K = 128 * 152 * 8, 256, 4096
    A = wl.make_matrix((M, K), 131, "int")
    B = wl.make_matrix((K, N), 132, "int")
    dA, dB = A.cuda(), B.cuda()
    lo, hi = torch.cuda.Stream(priority=0), torch.cuda.Stream(priority=-1)
    with m.Gemm(0) as g:
        C = torch.full((M, N), float("nan"), device="cuda")
        g.run(dA, dB, C, stream=lo)          # sizes the workspace
        torch.cuda.synchronize()
        C.fill_(float("nan"))
        torch.cuda.synchronize()
        g.run(dA, dB, C, stream=lo)
        g.occupy_start(24, limit_ns=20_000_000_000, stream=hi)
        try:
            lo.synchronize()
        finally:
            timed_out = g.occupy_stop()
        torch.cuda.synchronize()
        assert timed_out == 0
        g.sync(lo)
        ref = oracle.gemm(A, B)
        assert np.array_equal(C.cpu().numpy().astype(np.float64), ref)
        owner_lin, first = check_log(g, "clc", [M // 128], N // 256, 1)
