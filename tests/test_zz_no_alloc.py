"""gemm_run_noalloc: the GEMM for callers that cannot allocate device memory (a process
whose device memory belongs to its own pool allocator or sits under a hard cap, or a
latency-critical path that cannot afford a cudaMalloc).  Its scratch is a fixed device
array inside the library, shared by every call.

Checked through the C ABI on two calls in a row per case, against gemm_run (the
handle-based entry point) within the tolerance the other tests use and against the CPU
oracle, so the second call also shows that the scratch left behind by the first does not
leak into its result; gemm_noalloc_status reads back each call's error word (zero) and
ownership log (each tile computed once).  Self-contained: it passes alone in a fresh
process and after the other tests.  Collected last (file name) so a failure here cannot
hide others.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from oracle import within_tolerance
from oracle import coverage as cv
from tests.gpu_helpers import grid_of, linear_log

pytestmark = pytest.mark.gpu


def _reference(g, A, B, tile, cluster, sched):
    C = torch.full((A.shape[0], B.shape[1]), float("nan"), dtype=torch.float32, device="cuda")
    g.run(A, B, C, tile=tile, cluster=cluster, sched=sched)
    g.sync()
    return C.cpu().numpy()


def test_noalloc_matches_gemm_run_and_the_oracle_on_two_calls():
    import blackwell_clc_dynamic_gb300 as m

    cases = [
        # (M, N, K, tile, cluster, sched, seed): the first call covers more tiles than the
        # second, so stale scratch from call 1 would show up in call 2
        (1000, 776, 1000, (128, 256, 64), 1, "clc", 91),
        (384, 512, 256, (128, 128, 64), 1, "static", 92),
        (1000, 776, 1000, (128, 256, 64), (2, 2, 1), "clc", 93),
    ]
    with m.Gemm(0) as g:
        for M, N, K, tile, cl, sched, seed in cases:
            A_h = wl.make_matrix((M, K), seed)
            B_h = wl.make_matrix((K, N), seed + 100)
            A, B = A_h.cuda(), B_h.cuda()
            ref = _reference(g, A, B, tile, cl, sched)
            exact = oracle.gemm(A_h, B_h)
            mt, nt, ncta, rn = grid_of(M, N, tile, cl)
            for call in range(2):
                C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
                rc = m.gemm_run_noalloc(M, N, K, A, B, C, tile=tile, cluster=cl, sched=sched)
                assert rc == m.GEMM_OK, m.gemm_strerror(rc)
                # static launches one worker per SM (per cluster of SMs), the others one per tile
                sms = torch.cuda.get_device_properties(0).multi_processor_count
                n_workers = sms // ncta if sched == "static" else mt * nt
                rc, words, owner, claims, first = m.gemm_noalloc_status(mt * nt * ncta, n_workers)
                assert rc == m.GEMM_OK and words == (0, 0, 0), (rc, words)
                out = C.cpu().numpy()
                ok, worst = within_tolerance(out, ref.astype(np.float64))
                assert ok, f"call {call}: gemm_run_noalloc differs from gemm_run: worst ratio {worst:.3g}"
                ok, worst = within_tolerance(out, exact)
                assert ok, f"call {call}: gemm_run_noalloc differs from the oracle: worst ratio {worst:.3g}"
                owner_lin, claims_lin = linear_log(owner, claims, [mt], nt, ncta, group_rows=16, rn=rn)
                cv.check_device_log(sched, owner_lin, claims_lin, first.tolist(), n_workers,
                                    n_workers=n_workers if sched == "static" else None)
                # the log's sizes must be the latest call's
                rc, *_ = m.gemm_noalloc_status(mt * nt * ncta + 1, n_workers)
                assert rc == m.GEMM_ERR_INVALID_ARG


def test_noalloc_rejects_problems_beyond_its_scratch_and_host_memory():
    import blackwell_clc_dynamic_gb300 as m

    A = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((128, 256), dtype=torch.float32, device="cuda")
    # 65537 row tiles x 1 column tile: one tile more than the scratch holds; rejected
    # before anything is launched, so the small buffers are never touched
    rc = m.gemm_run_noalloc(128 * 65537, 256, 64, A, B, C)
    assert rc == m.GEMM_ERR_SCRATCH_LIMIT
    assert "scratch" in m.gemm_strerror(rc)
    # operands in pinned host memory: refused before any tensor map is made
    C_host = torch.zeros((128, 256), dtype=torch.float32).pin_memory()
    assert m.gemm_run_noalloc(128, 256, 64, A, B, C_host) == m.GEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()
