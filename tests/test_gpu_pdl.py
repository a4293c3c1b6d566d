"""Programmatic dependent launch: a GEMM launched with `pdl` may start its prologue while
the previous kernel on the stream still runs, but every access to global memory waits for
that kernel.  Checked through the data the launches share."""
import pytest
import torch

import oracle
import workloads as wl
from tests.gpu_helpers import TILE_256, assert_close, check_log

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cl,mc", [(1, 0), (2, 0), (4, 0)], ids=["c1", "c2pair", "c4mc"])
def test_pdl_orders_reads_after_the_previous_kernel(cl, mc):
    import blackwell_clc_dynamic_gb300 as m
    M, N, K = 1024, 768, 512
    A1 = wl.make_matrix((M, K), 111).cuda()
    B1 = wl.make_matrix((K, K), 112).cuda()
    B2 = wl.make_matrix((K, N), 113).cuda()
    with m.Gemm(0, pdl=True, cluster_b_multicast=mc) as g:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            C1 = torch.full((M, K), float("nan"), device="cuda")
            C2 = torch.full((M, N), float("nan"), device="cuda")
            for _ in range(3):
                g.run(A1, B1, C1, tile=TILE_256, cluster=cl, stream=s)
                A2 = C1.to(torch.bfloat16)            # a non-PDL kernel between the two GEMMs
                g.run(A2, B2, C2, tile=TILE_256, cluster=cl, stream=s)   # reads what it wrote
        s.synchronize()
        g.sync(s)
        A2h = A2.cpu()
        assert_close(C1.cpu().numpy(), oracle.gemm(A1.cpu(), B1.cpu()))
        assert_close(C2.cpu().numpy(), oracle.gemm(A2h, B2.cpu()))
        check_log(g, "clc", [-(-M // (128 * cl))], N // 256, cl)


def test_pdl_back_to_back_writes_keep_the_last_result():
    """Two PDL GEMMs writing the same C: the second's stores wait for the first kernel."""
    import blackwell_clc_dynamic_gb300 as m
    M, N, K = 2048, 1024, 1024
    A1 = wl.make_matrix((M, K), 121).cuda()
    A2 = wl.make_matrix((M, K), 122).cuda()
    B = wl.make_matrix((K, N), 123).cuda()
    with m.Gemm(0, pdl=True) as g:
        C = torch.full((M, N), float("nan"), device="cuda")
        for i in range(6):
            g.run(A1 if i % 2 == 0 else A2, B, C, sched=["clc", "static", "nonpersistent"][i % 3])
        g.sync()
        assert_close(C.cpu().numpy(), oracle.gemm(A2.cpu(), B.cpu()))
