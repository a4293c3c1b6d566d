"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element by element,
and the device ownership log against the coverage model (bit-exact invariants)."""

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from oracle import coverage as cv
from tests.gpu_helpers import (TILE_128, TILE_256, assert_close, check_log, cluster_dims, grid_of, rel_tolerance,
                               run)

pytestmark = pytest.mark.gpu

MODES = ["clc", "static", "nonpersistent"]
# (tile, cluster, B multicast): one CTA; CTA pair; clusters of 2 and 4 sharing B; 2 x 2
# clusters sharing A along rows and B along columns
C2X2 = (2, 2, 1)
SHAPES = [(TILE_256, 1, 0), (TILE_128, 1, 0), (TILE_256, 2, 0), (TILE_256, 2, 1), (TILE_256, 4, 0),
          (TILE_256, C2X2, 0)]
SHAPE_IDS = ["n256c1", "n128c1", "n256c2", "n256c2mc", "n256c4mc", "n256c2x2"]


@pytest.fixture(scope="module")
def g():
    import blackwell_clc_dynamic_gb300 as m
    h = m.Gemm(0)
    yield h
    h.close()


@pytest.fixture
def mc(g, request):
    """Selects B multicast for clusters of 2 for one test (from the `shape` parameter)."""
    flag = request.param
    g.set_opts(cluster_b_multicast=flag)
    yield flag
    g.set_opts(cluster_b_multicast=0)


def test_tiny_config_clc(g):
    """384x512x256, 128x128 tiles, 12 tiles, CLC over a grid of 12 CTAs."""
    w = wl.TINY
    A, B = wl.make_inputs(w)
    C = run(g, A, B, tile=TILE_128, cluster=1, sched="clc")
    assert_close(C, oracle.gemm(A, B))
    info = g.last_launch()
    assert info["grid_ctas"] == 12 and info["n_tiles"] == 12
    owner, claims, first = g.get_log()
    assert claims.tolist() == [1] * 12
    check_log(g, "clc", [3], 4, 1)


@pytest.mark.parametrize("tile,cl,mc", SHAPES, ids=SHAPE_IDS, indirect=["mc"])
@pytest.mark.parametrize("mode", MODES)
def test_integer_inputs_bit_exact(g, tile, cl, mc, mode):
    """Integer entries in [-4, 4]: every fp32 partial sum is an exact integer below 2^24,
    so any accumulation order must reproduce the oracle bit for bit."""
    M, N, K = 512, 768, 1024
    A = wl.make_matrix((M, K), 11, "int")
    B = wl.make_matrix((K, N), 12, "int")
    C = run(g, A, B, tile=tile, cluster=cl, sched=mode, num_workers=7)
    ref = oracle.gemm(A, B)
    assert np.array_equal(C.astype(np.float64), ref)


@pytest.mark.parametrize("tile,cl,mc", SHAPES, ids=SHAPE_IDS, indirect=["mc"])
@pytest.mark.parametrize("mode", MODES)
def test_uniform_ragged_tail(g, tile, cl, mc, mode):
    """Several tiles in each direction plus ragged M, N and K edges."""
    M, N, K = 1000, 776, 1000
    A = wl.make_matrix((M, K), 21)
    B = wl.make_matrix((K, N), 22)
    C = run(g, A, B, tile=tile, cluster=cl, sched=mode, num_workers=5)
    assert_close(C, oracle.gemm(A, B))
    mt, nt, ncta, rn = grid_of(M, N, tile, cl)
    check_log(g, mode, [mt], nt, ncta, num_workers=5 if mode == "static" else None, rn=rn)


def test_identity_and_rank_one(g):
    K = 256
    A = wl.make_matrix((384, K), 31)
    eye = torch.zeros((K, 512), dtype=torch.bfloat16)
    eye[torch.arange(K), torch.arange(K)] = 1
    C = run(g, A, eye)
    assert np.array_equal(C[:, :K], A.float().numpy()) and np.all(C[:, K:] == 0)
    u = torch.tensor([2.0 ** (i % 7 - 3) * (-1) ** i for i in range(256)])
    v = torch.tensor([2.0 ** (j % 5 - 2) * (-1) ** (j // 3) for j in range(512)])
    A1 = u[:, None].expand(256, K).contiguous().to(torch.bfloat16)
    B1 = v[None, :].expand(K, 512).contiguous().to(torch.bfloat16)
    C1 = run(g, A1, B1, sched="static")
    assert np.array_equal(C1.astype(np.float64), K * np.outer(u.double().numpy(), v.double().numpy()))


def test_empty_and_degenerate(g):
    # M == 0: nothing launched, no error
    A = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((0, 256), dtype=torch.float32, device="cuda")
    g.run(A, B, C)
    g.sync()
    assert g.last_launch()["launched"] == 0
    # K == 0: C = 0
    A = torch.zeros((200, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    C = torch.full((200, 256), float("nan"), device="cuda")
    g.run(A, B, C)
    g.sync()
    assert torch.all(C == 0)
    # a single tile, single row / column block
    A = wl.make_matrix((1, 64), 41)
    B = wl.make_matrix((64, 8), 42)
    assert_close(run(g, A, B), oracle.gemm(A, B))


def test_argument_errors(g):
    import blackwell_clc_dynamic_gb300 as m
    A = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((128, 256), dtype=torch.float32, device="cuda")
    h = g.h
    assert m.gemm_run(h, 128, 256, 64, A, B, C, tile=(128, 192, 64)) == m.GEMM_ERR_INVALID_ARG
    assert m.gemm_run(h, 128, 256, 64, A, B, C, tile=(128, 128, 64), cluster=2) == m.GEMM_ERR_INVALID_ARG
    assert m.gemm_run(h, 128, 256, 64, A, B, C, sched=7) == m.GEMM_ERR_INVALID_ARG
    assert m.gemm_run(h, 128, 256, 60, A, B, C) == m.GEMM_ERR_ALIGNMENT
    assert m.gemm_run(h, 128, 252, 64, A, B, C) == m.GEMM_ERR_ALIGNMENT
    assert m.gemm_run(h, 128, 256, 64, A.data_ptr() + 2, B, C) == m.GEMM_ERR_ALIGNMENT
    assert m.gemm_run(h, -1, 256, 64, A, B, C) == m.GEMM_ERR_INVALID_ARG
    assert m.gemm_run(h, 128, 256, 64, None, B, C) == m.GEMM_ERR_INVALID_ARG


def test_size_limits_and_empty_calls(g):
    """Sizes beyond 32-bit tile and row counts are refused before anything is allocated or
    launched; an empty grouped call and zero-sized problems are no-ops."""
    import blackwell_clc_dynamic_gb300 as m
    A = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((128, 256), dtype=torch.float32, device="cuda")
    h = g.h
    assert m.gemm_run(h, 1 << 31, 256, 64, A, B, C) == m.GEMM_ERR_TOO_LARGE
    assert m.gemm_run(h, 128, 1 << 31, 64, A, B, C) == m.GEMM_ERR_TOO_LARGE
    assert m.gemm_run(h, 128, 256, 1 << 31, A, B, C) == m.GEMM_ERR_TOO_LARGE
    assert m.gemm_run_grouped(h, [], 256, 64, [], [], []) == m.GEMM_OK
    assert m.gemm_run_grouped_v(h, [0, 0], [256, 256], [64, 64], [A, A], [B, B], [C, C]) == m.GEMM_OK
    assert m.gemm_run(h, 0, 256, 64, A, B, C) == m.GEMM_OK
    assert m.gemm_run(h, 128, 0, 64, A, B, C) == m.GEMM_OK
    g.sync()


def test_operands_must_be_memory_of_the_handles_device(g):
    """A, B and C must be device memory of the handle's GPU: pinned host memory (which the
    GPU could reach) is refused before any tensor map is encoded, for every entry point."""
    import blackwell_clc_dynamic_gb300 as m
    A = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((128, 256), dtype=torch.float32, device="cuda")
    Ah, Bh, Ch = A.cpu().pin_memory(), B.cpu().pin_memory(), C.cpu().pin_memory()
    h = g.h
    for args in ((Ah, B, C), (A, Bh, C), (A, B, Ch)):
        assert m.gemm_run(h, 128, 256, 64, *args) == m.GEMM_ERR_INVALID_ARG
    assert m.gemm_run_grouped(h, [128], 256, 64, [Ah], [B], [C]) == m.GEMM_ERR_INVALID_ARG
    assert m.gemm_run_grouped_v(h, [128], [256], [64], [A], [B], [Ch]) == m.GEMM_ERR_INVALID_ARG
    # the same operands in device memory run
    assert m.gemm_run(h, 128, 256, 64, A, B, C) == m.GEMM_OK
    assert m.gemm_run_grouped(h, [128], 256, 64, [A], [B], [C]) == m.GEMM_OK
    g.sync()


def test_handle_without_multicast_refuses_the_multicast_shapes():
    """A handle created with multicast = 0 (what every process of a multi-GPU job uses)
    never launches a kernel whose CTAs share operand tiles by TMA multicast; the CTA pair
    and one-CTA shapes still run."""
    import blackwell_clc_dynamic_gb300 as m
    A = wl.make_matrix((512, 256), 301, "int")
    B = wl.make_matrix((256, 512), 302, "int")
    with m.Gemm(0, multicast=False) as h:
        dA, dB = A.cuda(), B.cuda()
        C = torch.zeros((512, 512), dtype=torch.float32, device="cuda")
        for cl in (4, (2, 2, 1)):
            assert m.gemm_run(h.h, 512, 512, 256, dA, dB, C, cluster=cl) == m.GEMM_ERR_MULTICAST
        h.set_opts(cluster_b_multicast=1, multicast=1)      # multicast stays as created
        assert m.gemm_run(h.h, 512, 512, 256, dA, dB, C, cluster=2) == m.GEMM_ERR_MULTICAST
        with pytest.raises(m.GemmError):
            h.max_active_clusters(TILE_256, 4)
        h.set_opts(cluster_b_multicast=0)
        ref = oracle.gemm(A, B)
        for cl in (1, 2):
            assert np.array_equal(run(h, A, B, cluster=cl).astype(np.float64), ref)


@pytest.mark.parametrize("T", [1, 2, 5])
def test_static_owner_map_exact(g, T):
    """Static: tile t is run by worker t mod W, bit-exact; W above the tile count too."""
    M, N, K = 128 * 3 * T, 512, 128
    A = wl.make_matrix((M, K), 51)
    B = wl.make_matrix((K, N), 52)
    for W in (1, 4, 148):
        C = run(g, A, B, sched="static", num_workers=W)
        assert_close(C, oracle.gemm(A, B))
        owner_lin, first = check_log(g, "static", [3 * T], 2, 1, num_workers=W)
        assert owner_lin == cv.expected_owner_static(6 * T, W)


def test_log_keeps_only_the_latest_launch():
    """The device log is tagged per launch instead of cleared before it: entries of an
    earlier, larger launch on the same handle must not show through a later, smaller one,
    nor through a launch that ran with the log switched off."""
    import blackwell_clc_dynamic_gb300 as m
    h = m.Gemm(0)
    try:
        A = wl.make_matrix((128 * 8, 64), 71)
        B = wl.make_matrix((64, 256 * 8), 72)
        assert_close(run(h, A, B, sched="clc"), oracle.gemm(A, B))          # 64 tiles, 64 workers
        check_log(h, "clc", [8], 8, 1)
        a = wl.make_matrix((128 * 2, 64), 73)
        b = wl.make_matrix((64, 256 * 4), 74)
        assert_close(run(h, a, b, sched="static", num_workers=32), oracle.gemm(a, b))
        check_log(h, "static", [2], 4, 1, num_workers=32)                  # workers 8..31 never ran
        owner, claims, first = h.get_log()
        assert claims.tolist() == [1] * 8 and first[8:].tolist() == [-1] * 24
        h.set_opts(log_enable=0)
        run(h, A, B, sched="clc")
        h.set_opts(log_enable=1)
        with pytest.raises(m.GemmError):      # the most recent launch wrote no log
            h.get_log()
        assert_close(run(h, a, b, sched="nonpersistent"), oracle.gemm(a, b))
        check_log(h, "nonpersistent", [2], 4, 1)
        assert_close(run(h, A, B, sched="clc"), oracle.gemm(A, B))
        owner, claims, first = h.get_log()
        assert claims.tolist() == [1] * 64 and sorted(set(owner.tolist())) == sorted(set(first.tolist()) - {-1})
    finally:
        h.close()


@pytest.mark.parametrize("n_fetch", [0, 1, 5])
def test_clc_injected_failure_keeps_coverage(g, n_fetch):
    """After n successful fetches the scheduler reports a failed fetch without issuing a
    cancel; the workers stop and the launches nobody took run normally."""
    g.set_opts(inject_fail_after=n_fetch)
    try:
        M, N, K = 128 * 40, 512, 256
        A = wl.make_matrix((M, K), 61)
        B = wl.make_matrix((K, N), 62)
        C = run(g, A, B, sched="clc")
        assert_close(C, oracle.gemm(A, B))
        owner_lin, first = check_log(g, "clc", [40], 2, 1)
        counts = np.bincount(np.array(owner_lin), minlength=80)
        assert counts.max() <= n_fetch + 1
    finally:
        g.set_opts(inject_fail_after=-1)


@pytest.mark.parametrize("T", [147, 148, 149, 296, 297])
def test_tail_sweep_full(g, T):
    """Tail sweep workload (M = 128 T, N = 256, K = 8192, seed 2), CLC, static-persistent
    (148 workers) and non-persistent: every element of C against the oracle."""
    w = wl.tail(T)
    A, B = wl.make_inputs(w)
    dA, dB = A.cuda(), B.cuda()
    ref = oracle.gemm(A, B)
    for mode in MODES:
        C = torch.full((w.M, w.N), float("nan"), device="cuda")
        g.run(dA, dB, C, sched=mode, num_workers=148)
        g.sync()
        assert_close(C.cpu().numpy(), ref)
        check_log(g, mode, [T], 1, 1, num_workers=148 if mode == "static" else None)


@pytest.mark.parametrize("tile,cl,mc", SHAPES, ids=SHAPE_IDS, indirect=["mc"])
def test_grouped_small(g, tile, cl, mc):
    """Grouped flat grid over problems of uneven height (including an empty one)."""
    Ms = [128, 300, 0, 1024, 64]
    N, K = 512, 384
    gen = torch.Generator().manual_seed(71)
    As = [(torch.rand((m, K), generator=gen) * 2 - 1).to(torch.bfloat16) for m in Ms]
    Bs = [(torch.rand((K, N), generator=gen) * 2 - 1).to(torch.bfloat16) for _ in Ms]
    if True:
        for mode in MODES:
            dA = [a.cuda() for a in As]
            dB = [b.cuda() for b in Bs]
            dC = [torch.full((m, N), float("nan"), device="cuda") for m in Ms]
            g.run_grouped(dA, dB, dC, tile=tile, cluster=cl, sched=mode, num_workers=3)
            g.sync()
            for a, b, c in zip(As, Bs, dC):
                if a.shape[0]:
                    assert_close(c.cpu().numpy(), oracle.gemm(a, b))
            grids = [grid_of(m, N, tile, cl) for m in Ms]
            ncta, rn = grids[0][2], grids[0][3]
            check_log(g, mode, [gr[0] for gr in grids], grids[0][1], ncta,
                      num_workers=3 if mode == "static" else None, rn=rn)


def test_run_host_matches_device_run(g):
    A = wl.make_matrix((640, 512), 81)
    B = wl.make_matrix((512, 768), 82)
    Ch = torch.empty((640, 768), dtype=torch.float32).pin_memory()
    g.run_host(A.pin_memory(), B.pin_memory(), Ch)
    g.sync()
    assert_close(Ch.numpy(), oracle.gemm(A, B))


_INPUTS = {}
_REFS = {}


def _inputs(w):
    """Seeded inputs of a full-size workload, drawn once per test session (one workload
    held at a time)."""
    if w.name not in _INPUTS:
        _INPUTS.clear()
        _REFS.clear()
        _INPUTS[w.name] = wl.make_inputs(w)
    return _INPUTS[w.name]


def _reference(w):
    """The oracle's C of a full-size workload (every element, fp64; a list of per-problem
    results for grouped workloads), computed once and shared by the schedules compared
    with it."""
    A, B = _inputs(w)
    if w.name not in _REFS:
        _REFS[w.name] = [oracle.gemm(a, b) for a, b in zip(A, B)] if w.group_m else oracle.gemm(A, B)
    return _REFS[w.name]


def _full_check(C_dev, ref, K=0):
    """Every element of C against the oracle at the stated tolerance (scaled for products
    deeper than the stated workloads, see rel_tolerance); an element the kernel never wrote
    stays NaN and fails."""
    assert_close(C_dev.cpu().numpy(), ref, rel_tolerance(K))


@pytest.mark.parametrize("mode", MODES)
def test_square_full_size(g, mode):
    """M = N = K = 8192 (seed 1), 128 x 256 tiles, the bench's launch configuration: all of C
    against the oracle."""
    w = wl.SQUARE
    A, B = _inputs(w)
    ref = _reference(w)
    C = torch.full((w.M, w.N), float("nan"), device="cuda")
    g.run(A.cuda(), B.cuda(), C, sched=mode, num_workers=148)
    g.sync()
    _full_check(C, ref)
    check_log(g, mode, [64], 32, 1, num_workers=148 if mode == "static" else None)


@pytest.mark.parametrize("cl,mcast", [(2, 0), (2, 1), (4, 0), (C2X2, 0)],
                         ids=["pair", "c2_shared_b", "c4_shared_b", "c2x2_shared_ab"])
def test_square_full_size_cluster_modes(g, cl, mcast):
    """The square workload in the cluster launch configurations the benchmark times beside
    the headline (CLC): all of C against the oracle, exact log."""
    w = wl.SQUARE
    A, B = _inputs(w)
    ref = _reference(w)
    mt, nt, ncta, rn = grid_of(w.M, w.N, TILE_256, cl)
    g.set_opts(cluster_b_multicast=mcast)
    try:
        C = torch.full((w.M, w.N), float("nan"), device="cuda")
        g.run(A.cuda(), B.cuda(), C, cluster=cl, sched="clc")
        g.sync()
        _full_check(C, ref)
        check_log(g, "clc", [mt], nt, ncta, rn=rn)
    finally:
        g.set_opts(cluster_b_multicast=0)


@pytest.mark.parametrize("shape", ["square", "tail297", "pair"])
def test_clc_workers_steal(g, shape):
    """On an otherwise idle GPU with many more tiles than resident workers, CLC really takes
    work over ("CUTLASS CLC dynamic persistent kernel", section "What is cancelled is a
    launch, what is obtained is a work coordinate"): no more workers run than can be
    resident at once, workers run several tiles each, and the scheduler's trace names a
    successful try_cancel round trip for exactly the tiles that were not their own
    launch's, one per tile that no launch of its own computed (tiles - workers that ran)."""
    w = {"square": wl.SQUARE, "tail297": wl.tail(297), "pair": wl.PAIR}[shape]
    cl = 2 if shape == "pair" else 1
    A, B = _inputs(w) if shape == "square" else wl.make_inputs(w)
    mt, nt, ncta, rn = grid_of(w.M, w.N, TILE_256, cl)
    resident = g.max_active_clusters(TILE_256, cl)
    assert mt * nt > resident
    g.set_opts(trace_enable=1)
    try:
        C = torch.full((w.M, w.N), float("nan"), device="cuda")
        g.run(A.cuda(), B.cuda(), C, cluster=cl, sched="clc")
        g.sync()
        tr = g.get_trace().astype(np.int64)
    finally:
        g.set_opts(trace_enable=0)
    assert not torch.isnan(C).any()
    owner_lin, first = check_log(g, "clc", [mt], nt, ncta)
    T = mt * nt
    ran = sorted(set(owner_lin))
    counts = np.bincount(np.array(owner_lin), minlength=T)
    assert len(ran) <= resident, (len(ran), resident)
    assert counts.max() > 1 and counts[ran].min() >= 1
    stolen = np.array([owner_lin[t] != t for t in range(T)])
    assert stolen.sum() == T - len(ran)
    # round trips are recorded by rank 0's scheduler, on the CTA tile of rank 0 (cluster
    # tiles are row-major over CTA rows; rank r holds row block m * ncta + r)
    rt = np.zeros(T, dtype=np.int64)
    for c in range(T):
        m, n = cv.raster(c, mt, nt, g.opts.raster_group)
        rt[c] = tr[(m * ncta) * nt + n, 5]
    assert np.all(rt[stolen] > 0) and np.all(rt[~stolen] == 0)


@pytest.mark.parametrize("mode", MODES)
def test_pair_full_size_with_occupied_sms(g, mode):
    """M = N = 16384, K = 4096, normal(0, 0.02) (seed 3), 256 x 256 cluster tiles on CTA
    pairs, while an occupier kernel on another stream holds 24 SMs for the whole run: all
    of C against the oracle."""
    w = wl.PAIR
    A, B = _inputs(w)
    dA, dB = A.cuda(), B.cuda()
    C = torch.full((w.M, w.N), float("nan"), device="cuda")
    s_gemm = torch.cuda.Stream()
    s_occ = torch.cuda.Stream()
    # one unoccupied run first: it sizes the handle's log (growing the workspace
    # synchronises the device, which would wait for the occupier)
    g.run(dA, dB, C, cluster=2, sched=mode, num_workers=74)
    g.sync()
    C.fill_(float("nan"))
    torch.cuda.synchronize()
    g.occupy_start(24, limit_ns=20_000_000_000, stream=s_occ)
    try:
        g.occupy_wait_resident(10_000)
        g.run(dA, dB, C, cluster=2, sched=mode, num_workers=74, stream=s_gemm)
        s_gemm.synchronize()
    finally:
        timed_out = g.occupy_stop()
    torch.cuda.synchronize()
    assert timed_out == 0
    g.sync()
    _full_check(C, _reference(w))
    check_log(g, mode, [64], 64, 2, num_workers=74 if mode == "static" else None)


@pytest.mark.parametrize("mode", MODES)
def test_grouped_full_size(g, mode):
    """64 problems, N = K = 4096, M_g = 128 ceil(lognormal(2, 1)) clipped to [128, 8192]
    (seed 4), one flat grid of 12096 tiles of 128 x 256: every C_g in full."""
    w = wl.grouped()
    As, Bs = _inputs(w)
    dA = [a.cuda() for a in As]
    dB = [b.cuda() for b in Bs]
    dC = [torch.full((m, w.N), float("nan"), device="cuda") for m in w.group_m]
    g.run_grouped(dA, dB, dC, sched=mode, num_workers=148)
    g.sync()
    for c, ref in zip(dC, _reference(w)):
        _full_check(c, ref)
    check_log(g, mode, [m // 128 for m in w.group_m], 16, 1, num_workers=148 if mode == "static" else None)


@pytest.mark.parametrize("tile,cl,mc", SHAPES, ids=SHAPE_IDS, indirect=["mc"])
def test_run_host_banded_pipeline(g, tile, cl, mc):
    """gemm_run_host splits the product into blocks (2 row bands x 2 column bands here, the
    last of each ragged), copies them with strided copies and overlaps the copies with the
    block GEMMs on several streams; the result must equal the oracle."""
    M, N, K = 4200, 4104, 256
    A = wl.make_matrix((M, K), 83).pin_memory()
    B = wl.make_matrix((K, N), 84).pin_memory()
    Ch = torch.full((M, N), float("nan"), dtype=torch.float32).pin_memory()
    s = torch.cuda.Stream()
    g.run_host(A, B, Ch, tile=tile, cluster=cl, stream=s)
    s.synchronize()
    g.sync(s)
    assert_close(Ch.numpy(), oracle.gemm(A, B))


@pytest.mark.parametrize("tile,cl,mc", SHAPES, ids=SHAPE_IDS, indirect=["mc"])
@pytest.mark.parametrize("mode", MODES)
def test_grouped_varied_shapes_small(g, tile, cl, mc, mode):
    """Problems of different M, N and K in one flat grid (ragged edges, an empty problem,
    a K = 0 problem whose C must be zero)."""
    shapes = [(300, 520, 192), (128, 256, 1000), (0, 256, 64), (700, 264, 64), (256, 776, 0), (64, 1024, 512)]
    gen = torch.Generator().manual_seed(73)
    As = [(torch.rand((m, k), generator=gen) * 2 - 1).to(torch.bfloat16) for m, n, k in shapes]
    Bs = [(torch.rand((k, n), generator=gen) * 2 - 1).to(torch.bfloat16) for m, n, k in shapes]
    dC = [torch.full((m, n), float("nan"), device="cuda") for m, n, k in shapes]
    g.run_grouped_v([a.cuda() for a in As], [b.cuda() for b in Bs], dC, tile=tile, cluster=cl, sched=mode,
                    num_workers=3)
    g.sync()
    for (m, n, k), a, b, c in zip(shapes, As, Bs, dC):
        if m and n:
            ref = oracle.gemm(a, b) if k else np.zeros((m, n))
            assert_close(c.cpu().numpy(), ref)
    grids = [grid_of(m, n, tile, cl) for m, n, k in shapes if m and n]
    check_log(g, mode, [gr[0] for gr in grids], [gr[1] for gr in grids], grids[0][2],
              num_workers=3 if mode == "static" else None, rn=grids[0][3])


@pytest.mark.parametrize("mode", MODES)
def test_deep_products_bit_exact(g, mode):
    """Integer entries in [-4, 4] at depths up to 16384 (the varied-depth workload's clip):
    every partial sum stays below 2^18, exact in fp32 however the tensor cores align and
    round, so the result must equal the oracle bit for bit.  This pins the deep-K paths
    (plain and grouped, every schedule) apart from floating-point rounding."""
    shapes = [(256, 512, 16384), (130, 264, 12800), (384, 256, 8200), (128, 1024, 9000)]
    As = [wl.make_matrix((m, k), 400 + i, "int") for i, (m, n, k) in enumerate(shapes)]
    Bs = [wl.make_matrix((k, n), 500 + i, "int") for i, (m, n, k) in enumerate(shapes)]
    refs = [oracle.gemm(a, b) for a, b in zip(As, Bs)]
    dC = [torch.full((m, n), float("nan"), device="cuda") for m, n, k in shapes]
    g.run_grouped_v([a.cuda() for a in As], [b.cuda() for b in Bs], dC, sched=mode, num_workers=5)
    g.sync()
    for c, ref in zip(dC, refs):
        assert np.array_equal(c.cpu().numpy().astype(np.float64), ref)
    C = run(g, As[0], Bs[0], sched=mode, num_workers=5)
    assert np.array_equal(C.astype(np.float64), refs[0])


@pytest.mark.parametrize("mode", MODES)
def test_grouped_varied_depth_full_size(g, mode):
    """64 problems with K_g = 256 ceil(lognormal(2, 1)) in [256, 16384] and M_g as in the
    grouped workload (seed 5), N = 4096: tiles of unequal cost in one flat grid; every C_g
    in full."""
    w = wl.grouped_varied_depth()
    As, Bs = _inputs(w)
    dA = [a.cuda() for a in As]
    dB = [b.cuda() for b in Bs]
    dC = [torch.full((m, w.N), float("nan"), device="cuda") for m in w.group_m]
    g.run_grouped_v(dA, dB, dC, sched=mode, num_workers=148)
    g.sync()
    for c, ref, k in zip(dC, _reference(w), w.depths()):
        _full_check(c, ref, k)
    check_log(g, mode, [m // 128 for m in w.group_m], 16, 1, num_workers=148 if mode == "static" else None)


@pytest.mark.parametrize("dT", ["1", "sms-1", "sms", "sms+1", "2sms+1"])
@pytest.mark.parametrize("mode", ["clc", "static"])
def test_tile_count_around_the_sm_count(g, dT, mode):
    """Fewer, as many and slightly more tiles than resident workers, relative to the queried
    SM count: coverage stays exact and static workers follow t mod W."""
    sms = g.sm_count
    T = {"1": 1, "sms-1": sms - 1, "sms": sms, "sms+1": sms + 1, "2sms+1": 2 * sms + 1}[dT]
    M, N, K = 128 * T, 256, 512
    A = wl.make_matrix((M, K), 141, "int")
    B = wl.make_matrix((K, N), 142, "int")
    C = run(g, A, B, sched=mode, num_workers=sms)
    assert np.array_equal(C.astype(np.float64), oracle.gemm(A, B))
    owner_lin, first = check_log(g, mode, [T], 1, 1, num_workers=sms if mode == "static" else None)
    if mode == "static":
        assert owner_lin == cv.expected_owner_static(T, sms)
    else:
        # at most one worker per resident slot plus the launches nobody took
        assert len(set(owner_lin)) <= T


def test_randomized_shapes_and_modes(g):
    """24 seeded random problems: ragged M, N, K (multiples of 8 where the ABI needs it),
    every schedule and cluster shape, integer inputs so the result must be bit-exact."""
    rng = np.random.default_rng(2024)
    try:
        for i in range(24):
            tile, cl, mcast = SHAPES[i % len(SHAPES)]
            mode = MODES[(i // len(SHAPES)) % 3]
            M = int(rng.integers(1, 1500))
            N = 8 * int(rng.integers(1, 160))
            K = 8 * int(rng.integers(0, 200))
            A = wl.make_matrix((M, K), 1000 + i, "int")
            B = wl.make_matrix((K, N), 2000 + i, "int")
            g.set_opts(cluster_b_multicast=mcast, raster_group=int(rng.integers(1, 17)))
            C = run(g, A, B, tile=tile, cluster=cl, sched=mode, num_workers=int(rng.integers(1, 300)))
            ref = oracle.gemm(A, B) if K else np.zeros((M, N))
            assert np.array_equal(C.astype(np.float64), ref), (i, M, N, K, tile, cl, mcast, mode)
    finally:
        g.set_opts(cluster_b_multicast=0, raster_group=16)


@pytest.mark.parametrize("cl,mcast,mode", [(1, 0, "clc"), (1, 0, "static"), (2, 0, "clc"), (4, 0, "clc"),
                                           (C2X2, 0, "clc")],
                         ids=["c1-clc", "c1-static", "pair-clc", "c4-clc", "c2x2-clc"])
def test_trace_is_consistent_with_the_log(g, cl, mcast, mode):
    """Per tile: producer start <= last MMA issued <= epilogue start <= last store issued;
    the SM id is below the SM count; the worker is the one the ownership log names; CLC
    round trips are recorded only for tiles that came from a cancel."""
    ncta, rm, rn = cluster_dims(cl)
    M, N, K = 128 * rm * 40, 512, 1024
    A = wl.make_matrix((M, K), 151)
    B = wl.make_matrix((K, N), 152)
    g.set_opts(trace_enable=1, cluster_b_multicast=mcast)
    try:
        C = run(g, A, B, cluster=cl, sched=mode, num_workers=37)
        tr = g.get_trace().astype(np.int64)
        owner, claims, first = g.get_log()
    finally:
        g.set_opts(trace_enable=0, cluster_b_multicast=0)
    assert_close(C, oracle.gemm(A, B))
    start, end, sm, worker, wait, rt, epi, last_mma = (tr[:, i] for i in range(8))
    assert np.all(start > 0) and np.all(end >= start) and np.all(epi >= start) and np.all(end >= epi)
    # CTA tiles are row-major over (M/128) x (N/256); the CTA of rank r holds row block
    # rm*m + r // rn and column block rn*n + r % rn.  The MMA time is recorded by the CTA
    # that issues the MMA: every CTA, or rank 0 of a CTA pair.
    pos = np.arange(len(tr))
    rank = ((pos // (N // 256)) % rm) * rn + (pos % (N // 256)) % rn
    issuer = np.ones(len(tr), dtype=bool) if (ncta == 1 or mcast or ncta == 4) else rank == 0
    assert np.all(last_mma[issuer] >= start[issuer]) and np.all(epi[issuer] >= last_mma[issuer])
    assert np.all(sm < g.sm_count)
    assert np.array_equal(worker, owner.astype(np.int64))
    if mode == "static":
        assert np.all(rt == 0)
    else:
        # round trips are written by the scheduler of rank 0 for the tiles its cancels
        # returned; a worker's own first tile has none
        assert np.all(rt[rank != 0] == 0)


@pytest.mark.parametrize("ahead", [1, 2])
@pytest.mark.parametrize("cl", [1, 2, C2X2], ids=["c1", "pair", "c2x2"])
def test_fetch_ahead_keeps_coverage(g, ahead, cl):
    """With extra throttle tokens a worker holds up to 1 + ahead fetched tiles; results and
    coverage do not change."""
    ncta, rm, rn = cluster_dims(cl)
    M, N, K = 128 * rm * 50, 512 * rn, 512
    A = wl.make_matrix((M, K), 181, "int")
    B = wl.make_matrix((K, N), 182, "int")
    g.set_opts(fetch_ahead=ahead)
    try:
        C = run(g, A, B, cluster=cl, sched="clc")
    finally:
        g.set_opts(fetch_ahead=0)
    assert np.array_equal(C.astype(np.float64), oracle.gemm(A, B))
    check_log(g, "clc", [50], 2, ncta, rn=rn)


@pytest.mark.parametrize("cl", [1, 2, C2X2], ids=["c1", "pair", "c2x2"])
def test_l2_prefetch_option_keeps_results(g, cl):
    """The optional L2 prefetch ahead of the ring (a hint: it moves no data into shared
    memory) leaves results and coverage unchanged, ragged edges included."""
    ncta, rm, rn = cluster_dims(cl)
    M, N, K = 1000, 776, 2040
    A = wl.make_matrix((M, K), 201, "int")
    B = wl.make_matrix((K, N), 202, "int")
    g.set_opts(l2_prefetch=8)
    try:
        C = run(g, A, B, cluster=cl, sched="clc")
    finally:
        g.set_opts(l2_prefetch=0)
    assert np.array_equal(C.astype(np.float64), oracle.gemm(A, B))
    mt, nt, ncta, rn = grid_of(M, N, TILE_256, cl)
    check_log(g, "clc", [mt], nt, ncta, rn=rn)
