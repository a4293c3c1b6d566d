"""The C-ABI library loads and exports every symbol include/clcgemm.h declares (no GPU
needed); host-side behaviour that needs no device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "clcgemm.h")


@pytest.fixture(scope="module")
def pkg():
    import __graft_entry__
    __graft_entry__._load_build_module().build()
    import blackwell_clc_dynamic_gb300 as m
    return m


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"CLCGEMM_API\s+[\w\s\*]*?\b(gemm_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gemm_create", "gemm_run", "gemm_destroy", "gemm_run_grouped", "gemm_get_log",
                     "gemm_sync", "gemm_strerror"):
        assert required in names


def test_every_declared_symbol_is_exported(pkg):
    lib = ctypes.CDLL(pkg.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(pkg.EXPORTS) == declared_functions()


def test_no_cuda_types_in_signatures():
    text = open(HEADER).read()
    for banned in ("cudaStream_t", "CUtensorMap", "torch", "at::"):
        assert banned not in re.sub(r"/\*.*?\*/", "", text, flags=re.S)


def test_strerror_and_version(pkg):
    assert pkg.gemm_strerror(0) == "ok"
    assert "alignment" in pkg.gemm_strerror(pkg.GEMM_ERR_ALIGNMENT)
    assert pkg.gemm_strerror(12345) == "unknown error"
    assert pkg.gemm_version() == 100


def test_opts_default(pkg):
    o = pkg.gemm_opts_default()
    assert (o.log_enable, o.trace_enable, o.timeout_ns, o.inject_fail_after, o.raster_group, o.l2_prefetch,
            o.hold_scheduler, o.cluster_b_multicast, o.pdl, o.fetch_ahead,
            o.multicast) == (1, 0, 2_000_000_000, -1, 16, 0, 0, 0, 0, 0, 1)


def test_create_without_gpu_reports_no_device(pkg):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, h = pkg.gemm_create(0)
    assert rc == pkg.GEMM_ERR_NO_DEVICE and h is None


def test_checked_build_exports_the_same_symbols(pkg):
    """The bounds-checked build (CLCG_BOUNDS_CHECK) is the same library with checks added."""
    import __graft_entry__
    path = __graft_entry__._load_build_module().build(checked=True)
    lib = ctypes.CDLL(path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_new_error_codes_are_named(pkg):
    assert "multicast" in pkg.gemm_strerror(pkg.GEMM_ERR_MULTICAST)
    assert "bounds" in pkg.gemm_strerror(pkg.GEMM_ERR_BOUNDS)


def test_noalloc_status_without_device(pkg):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, words, owner, claims, first = pkg.gemm_noalloc_status(0, 0)
    assert rc == pkg.GEMM_ERR_NO_DEVICE


def test_null_handle_is_rejected(pkg):
    assert pkg.lib.gemm_run(None, 128, 256, 64, None, None, None, pkg.gemm_tile_t(128, 256, 64),
                            pkg.gemm_cluster_t(1, 1, 1), 0, 0, None) == pkg.GEMM_ERR_INVALID_ARG
    assert pkg.lib.gemm_sync(None, None) == pkg.GEMM_ERR_INVALID_ARG
    pkg.gemm_destroy(None)
