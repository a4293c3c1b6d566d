"""Repeated launches: a race in the CLC response ring, the throttle or the operand ring
would show up as a wrong element or a tile claimed twice or never in some launch.  Integer
inputs make every correct result bit-identical to the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

CASES = [  # (M, N, K, tile, cluster, B multicast)
    (1536, 1024, 1024, (128, 256, 64), 1, 0),
    (1408, 768, 640, (128, 128, 64), 1, 0),
    (2048, 1024, 512, (128, 256, 64), 2, 0),
    (2048, 1024, 512, (128, 256, 64), 2, 1),
    (4096, 512, 512, (128, 256, 64), 4, 0),
]


@pytest.mark.parametrize("case", range(len(CASES)), ids=["c1n256", "c1n128", "pair", "c2mc", "c4mc"])
def test_many_launches_stay_exact(case):
    import blackwell_clc_dynamic_gb300 as m
    M, N, K, tile, cl, mcast = CASES[case]
    A = wl.make_matrix((M, K), 161 + case, "int")
    B = wl.make_matrix((K, N), 171 + case, "int")
    ref = oracle.gemm(A, B).astype(np.float32)
    dA, dB = A.cuda(), B.cuda()
    dref = torch.from_numpy(ref).cuda()
    with m.Gemm(0, cluster_b_multicast=mcast) as g:
        C = torch.empty((M, N), dtype=torch.float32, device="cuda")
        for i in range(60):
            sched = ("clc", "clc", "static", "clc", "nonpersistent")[i % 5]
            C.fill_(float("nan"))
            g.run(dA, dB, C, tile=tile, cluster=cl, sched=sched, num_workers=(i * 7) % 150 + 1)
            g.sync()
            assert torch.equal(C, dref), f"launch {i} ({sched}) differs"
            owner, claims, first = g.get_log()
            assert np.all(claims == 1), f"launch {i} ({sched}): claims {np.unique(claims)}"
