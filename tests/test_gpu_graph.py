"""CUDA-graph capture of gemm_run: launches captured once and replayed reproduce the
oracle's result, for one-CTA, CTA-pair and 2 x 2 cluster launches and for the CLC and
static schedules.  The ownership log is switched off for capture: a replay reuses the
launch tag it was captured with, so a replayed launch's log entries would not be its own."""
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_helpers import assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cluster", [1, 2, (2, 2, 1)], ids=["c1", "pair", "c2x2"])
def test_captured_launches_replay_correctly(cluster):
    import blackwell_clc_dynamic_gb300 as m
    A = wl.make_matrix((1000, 512), 191)
    A2 = wl.make_matrix((640, 512), 193)
    B = wl.make_matrix((512, 776), 192)
    dA, dA2, dB = A.cuda(), A2.cuda(), B.cuda()
    ref, ref2 = oracle.gemm(A, B), oracle.gemm(A2, B)
    with m.Gemm(0, log=False) as g:
        C = torch.full((1000, 776), float("nan"), device="cuda")
        C2 = torch.full((640, 776), float("nan"), device="cuda")
        g.run(dA, dB, C, cluster=cluster)          # first use outside the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            g.run(dA, dB, C, cluster=cluster)
            g.run(dA2, dB, C2, cluster=cluster, sched="static", num_workers=5)
        for _ in range(2):
            C.fill_(float("nan"))
            C2.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            assert_close(C.cpu().numpy(), ref)
            assert_close(C2.cpu().numpy(), ref2)
        g.sync()
