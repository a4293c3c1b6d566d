"""Python binding of libclcgemm (the C ABI in include/clcgemm.h).

Argument marshalling only: every computation runs in the library's CUDA kernels.  The
module-level functions carry the C names (``gemm_create``, ``gemm_run``, ...); the
``Gemm`` class wraps a handle for convenience.  Torch tensors are accepted wherever the C
call takes a device or host pointer; PyTorch supplies memory and streams, nothing else.

Importing works without a GPU (the library loads and reports GEMM_ERR_NO_DEVICE on
use); a missing library is an ImportError, never a silent fallback.  With the
environment variable CLCGEMM_CHECKED=1 the bounds-checked build (libclcgemm_checked.so,
``build.py --checked``) is loaded instead.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

_HERE = os.path.dirname(os.path.abspath(__file__))
CHECKED = os.environ.get("CLCGEMM_CHECKED", "0") == "1"
LIB_PATH = os.path.join(_HERE, "libclcgemm_checked.so" if CHECKED else "libclcgemm.so")

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = -1
GEMM_ERR_UNSUPPORTED_DEVICE = -2
GEMM_ERR_ALIGNMENT = -3
GEMM_ERR_LAUNCH = -4
GEMM_ERR_TIMEOUT = -5
GEMM_ERR_OOM = -6
GEMM_ERR_CUDA = -7
GEMM_ERR_NO_DEVICE = -8
GEMM_ERR_TOO_LARGE = -9
GEMM_ERR_SCRATCH_LIMIT = -10
GEMM_ERR_MULTICAST = -11
GEMM_ERR_BOUNDS = -12

GEMM_SCHED_CLC = 0
GEMM_SCHED_STATIC = 1
GEMM_SCHED_NONPERSISTENT = 2
SCHED = {"clc": GEMM_SCHED_CLC, "static": GEMM_SCHED_STATIC, "nonpersistent": GEMM_SCHED_NONPERSISTENT}

# Every entry point declared in include/clcgemm.h.
EXPORTS = (
    "gemm_opts_default", "gemm_create", "gemm_destroy", "gemm_set_opts", "gemm_run", "gemm_run_grouped",
    "gemm_run_host", "gemm_sync", "gemm_device_error", "gemm_last_launch", "gemm_get_log", "gemm_get_trace",
    "gemm_max_active_clusters", "gemm_sm_count", "gemm_occupy_start", "gemm_occupy_wait_resident",
    "gemm_occupy_stop", "gemm_strerror", "gemm_version", "gemm_run_noalloc", "gemm_run_grouped_v",
    "gemm_noalloc_status",
)


class gemm_tile_t(ctypes.Structure):
    _fields_ = [("bm", ctypes.c_int), ("bn", ctypes.c_int), ("bk", ctypes.c_int)]


class gemm_cluster_t(ctypes.Structure):
    _fields_ = [("x", ctypes.c_int), ("y", ctypes.c_int), ("z", ctypes.c_int)]


class gemm_opts_t(ctypes.Structure):
    _fields_ = [("log_enable", ctypes.c_int), ("trace_enable", ctypes.c_int), ("timeout_ns", ctypes.c_int64),
                ("inject_fail_after", ctypes.c_int), ("raster_group", ctypes.c_int), ("l2_prefetch", ctypes.c_int),
                ("hold_scheduler", ctypes.c_int), ("cluster_b_multicast", ctypes.c_int), ("pdl", ctypes.c_int),
                ("fetch_ahead", ctypes.c_int), ("multicast", ctypes.c_int)]


class gemm_launch_info_t(ctypes.Structure):
    _fields_ = [("n_tiles", ctypes.c_int64), ("n_cluster_tiles", ctypes.c_int64), ("n_workers", ctypes.c_int64),
                ("grid_ctas", ctypes.c_int64), ("smem_bytes", ctypes.c_int), ("cluster", ctypes.c_int),
                ("sched", ctypes.c_int), ("launched", ctypes.c_int)]


class GemmError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {gemm_strerror(code)} ({code})" if what else f"{gemm_strerror(code)} ({code})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{os.path.basename(LIB_PATH)} is not built ({LIB_PATH}); run "
                          f"blackwell_clc_dynamic_gb300/build.py{' --checked' if CHECKED else ''}")
    lib = ctypes.CDLL(LIB_PATH)
    H = ctypes.c_void_p
    i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    sig = {
        "gemm_opts_default": (None, [ctypes.POINTER(gemm_opts_t)]),
        "gemm_create": (i32, [i32, ctypes.POINTER(gemm_opts_t), ctypes.POINTER(H)]),
        "gemm_destroy": (None, [H]),
        "gemm_set_opts": (i32, [H, ctypes.POINTER(gemm_opts_t)]),
        "gemm_run": (i32, [H, i64, i64, i64, p, p, p, gemm_tile_t, gemm_cluster_t, i32, i32, p]),
        "gemm_run_grouped": (i32, [H, i32, ctypes.POINTER(i64), i64, i64, ctypes.POINTER(p), ctypes.POINTER(p),
                                   ctypes.POINTER(p), gemm_tile_t, gemm_cluster_t, i32, i32, p]),
        "gemm_run_grouped_v": (i32, [H, i32, ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(i64),
                                     ctypes.POINTER(p), ctypes.POINTER(p), ctypes.POINTER(p), gemm_tile_t,
                                     gemm_cluster_t, i32, i32, p]),
        "gemm_run_host": (i32, [H, i64, i64, i64, p, p, p, gemm_tile_t, gemm_cluster_t, i32, i32, p]),
        "gemm_sync": (i32, [H, p]),
        "gemm_device_error": (i32, [H, ctypes.POINTER(ctypes.c_int32)]),
        "gemm_last_launch": (i32, [H, ctypes.POINTER(gemm_launch_info_t)]),
        "gemm_get_log": (i32, [H, p, p, p, i64, i64]),
        "gemm_get_trace": (i32, [H, p, i64]),
        "gemm_max_active_clusters": (i32, [H, gemm_tile_t, gemm_cluster_t, ctypes.POINTER(i32)]),
        "gemm_sm_count": (i32, [H, ctypes.POINTER(i32)]),
        "gemm_occupy_start": (i32, [H, i32, i64, p]),
        "gemm_occupy_wait_resident": (i32, [H, i32]),
        "gemm_occupy_stop": (i32, [H, ctypes.POINTER(i32)]),
        "gemm_strerror": (ctypes.c_char_p, [i32]),
        "gemm_version": (i32, []),
        "gemm_run_noalloc": (i32, [i64, i64, i64, p, p, p, gemm_tile_t, gemm_cluster_t, i32, i32, p]),
        "gemm_noalloc_status": (i32, [ctypes.POINTER(ctypes.c_int32), p, p, p, i64, i64, p]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()


# ------------------------------------------------------------------ marshalling helpers
def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(s) -> Optional[int]:
    if s is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except Exception:
            pass
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _tile(t) -> gemm_tile_t:
    return t if isinstance(t, gemm_tile_t) else gemm_tile_t(*t)


def _cluster(c) -> gemm_cluster_t:
    if isinstance(c, gemm_cluster_t):
        return c
    if isinstance(c, int):
        return gemm_cluster_t(c, 1, 1)
    return gemm_cluster_t(*c)


def _sched(s) -> int:
    return SCHED[s] if isinstance(s, str) else int(s)


def _check(rc: int, what: str) -> None:
    if rc != GEMM_OK:
        raise GemmError(rc, what)


# ------------------------------------------------------------------ C-named functions
def gemm_strerror(code: int) -> str:
    return lib.gemm_strerror(code).decode()


def gemm_version() -> int:
    return lib.gemm_version()


def gemm_opts_default() -> gemm_opts_t:
    o = gemm_opts_t()
    lib.gemm_opts_default(ctypes.byref(o))
    return o


def gemm_create(device: int = 0, opts: Optional[gemm_opts_t] = None) -> Tuple[int, Optional[int]]:
    h = ctypes.c_void_p()
    rc = lib.gemm_create(device, ctypes.byref(opts) if opts is not None else None, ctypes.byref(h))
    return rc, h.value


def gemm_destroy(h: int) -> None:
    lib.gemm_destroy(h)


def gemm_run(h, M, N, K, A, B, C, tile=(128, 256, 64), cluster=1, sched="clc", num_workers=0, stream=None) -> int:
    return lib.gemm_run(h, M, N, K, _ptr(A), _ptr(B), _ptr(C), _tile(tile), _cluster(cluster), _sched(sched),
                        num_workers, _stream(stream))


def gemm_run_host(h, M, N, K, A, B, C, tile=(128, 256, 64), cluster=1, sched="clc", num_workers=0,
                  stream=None) -> int:
    return lib.gemm_run_host(h, M, N, K, _ptr(A), _ptr(B), _ptr(C), _tile(tile), _cluster(cluster), _sched(sched),
                             num_workers, _stream(stream))


def gemm_run_grouped(h, M_g: Sequence[int], N, K, A_g, B_g, C_g, tile=(128, 256, 64), cluster=1, sched="clc",
                     num_workers=0, stream=None) -> int:
    G = len(M_g)
    m = (ctypes.c_int64 * G)(*M_g)
    a = (ctypes.c_void_p * G)(*[_ptr(x) for x in A_g])
    b = (ctypes.c_void_p * G)(*[_ptr(x) for x in B_g])
    c = (ctypes.c_void_p * G)(*[_ptr(x) for x in C_g])
    return lib.gemm_run_grouped(h, G, m, N, K, a, b, c, _tile(tile), _cluster(cluster), _sched(sched),
                                num_workers, _stream(stream))


def gemm_run_noalloc(M, N, K, A, B, C, tile=(128, 256, 64), cluster=1, sched="clc", num_workers=0,
                     stream=None) -> int:
    """gemm_run without a handle and without any device allocation (fixed scratch; see the
    C header for its limits and sharing rules)."""
    return lib.gemm_run_noalloc(M, N, K, _ptr(A), _ptr(B), _ptr(C), _tile(tile), _cluster(cluster), _sched(sched),
                                num_workers, _stream(stream))


def gemm_noalloc_status(n_tiles: int, n_workers: int, stream=None):
    """(rc, (bits, site, block), owner, claims, first) of the latest gemm_run_noalloc call on
    the current device: its device error word and ownership log (see the C header)."""
    import numpy as np
    w = (ctypes.c_int32 * 3)()
    owner = np.empty(n_tiles, dtype=np.int32)
    claims = np.empty(n_tiles, dtype=np.int32)
    first = np.empty(n_workers, dtype=np.int32)
    rc = lib.gemm_noalloc_status(w, owner.ctypes.data, claims.ctypes.data, first.ctypes.data, n_tiles, n_workers,
                                 _stream(stream))
    return rc, tuple(w), owner, claims, first


def gemm_run_grouped_v(h, M_g: Sequence[int], N_g: Sequence[int], K_g: Sequence[int], A_g, B_g, C_g,
                       tile=(128, 256, 64), cluster=1, sched="clc", num_workers=0, stream=None) -> int:
    G = len(M_g)
    m = (ctypes.c_int64 * G)(*M_g)
    n = (ctypes.c_int64 * G)(*N_g)
    k = (ctypes.c_int64 * G)(*K_g)
    a = (ctypes.c_void_p * G)(*[_ptr(x) for x in A_g])
    b = (ctypes.c_void_p * G)(*[_ptr(x) for x in B_g])
    c = (ctypes.c_void_p * G)(*[_ptr(x) for x in C_g])
    return lib.gemm_run_grouped_v(h, G, m, n, k, a, b, c, _tile(tile), _cluster(cluster), _sched(sched),
                                  num_workers, _stream(stream))


def gemm_sync(h, stream=None) -> int:
    return lib.gemm_sync(h, _stream(stream))


# ------------------------------------------------------------------ handle wrapper
class Gemm:
    """One library handle on one device."""

    def __init__(self, device: int = 0, log: bool = True, trace: bool = False, timeout_ns: int = 0,
                 inject_fail_after: int = -1, raster_group: int = 16, l2_prefetch: int = -1,
                 hold_scheduler: bool = False, cluster_b_multicast: bool = False, pdl: bool = False,
                 fetch_ahead: int = 0, multicast: bool = True):
        self.opts = gemm_opts_t(int(log), int(trace), int(timeout_ns), int(inject_fail_after), int(raster_group),
                                int(l2_prefetch), int(hold_scheduler), int(cluster_b_multicast), int(pdl),
                                int(fetch_ahead), int(multicast))
        rc, h = gemm_create(device, self.opts)
        _check(rc, "gemm_create")
        self.h = h
        self.device = device

    def close(self) -> None:
        if getattr(self, "h", None):
            gemm_destroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_opts(self, **kw) -> None:
        for k, v in kw.items():
            setattr(self.opts, k, int(v))
        _check(lib.gemm_set_opts(self.h, ctypes.byref(self.opts)), "gemm_set_opts")

    def run(self, A, B, C, tile=(128, 256, 64), cluster=1, sched="clc", num_workers=0, stream=None) -> None:
        M, K = A.shape
        N = B.shape[1]
        _check(gemm_run(self.h, M, N, K, A, B, C, tile, cluster, sched, num_workers, stream), "gemm_run")

    def run_host(self, A, B, C, tile=(128, 256, 64), cluster=1, sched="clc", num_workers=0, stream=None) -> None:
        M, K = A.shape
        N = B.shape[1]
        _check(gemm_run_host(self.h, M, N, K, A, B, C, tile, cluster, sched, num_workers, stream), "gemm_run_host")

    def run_grouped(self, As, Bs, Cs, tile=(128, 256, 64), cluster=1, sched="clc", num_workers=0,
                    stream=None) -> None:
        M_g = [a.shape[0] for a in As]
        K = As[0].shape[1] if As else 0
        N = Bs[0].shape[1] if Bs else 0
        _check(gemm_run_grouped(self.h, M_g, N, K, As, Bs, Cs, tile, cluster, sched, num_workers, stream),
               "gemm_run_grouped")

    def run_grouped_v(self, As, Bs, Cs, tile=(128, 256, 64), cluster=1, sched="clc", num_workers=0,
                      stream=None) -> None:
        """Problems of different shapes: C_g = A_g @ B_g with A_g (M_g x K_g), B_g (K_g x N_g)."""
        M_g = [a.shape[0] for a in As]
        K_g = [a.shape[1] for a in As]
        N_g = [b.shape[1] for b in Bs]
        _check(gemm_run_grouped_v(self.h, M_g, N_g, K_g, As, Bs, Cs, tile, cluster, sched, num_workers, stream),
               "gemm_run_grouped_v")

    def sync(self, stream=None) -> None:
        _check(gemm_sync(self.h, stream), "gemm_sync")

    def device_error(self) -> Tuple[int, int, int]:
        w = (ctypes.c_int32 * 3)()
        _check(lib.gemm_device_error(self.h, w), "gemm_device_error")
        return tuple(w)

    def last_launch(self) -> dict:
        info = gemm_launch_info_t()
        _check(lib.gemm_last_launch(self.h, ctypes.byref(info)), "gemm_last_launch")
        return {f: getattr(info, f) for f, _ in gemm_launch_info_t._fields_}

    def get_log(self):
        import numpy as np
        info = self.last_launch()
        owner = np.empty(info["n_tiles"], dtype=np.int32)
        claims = np.empty(info["n_tiles"], dtype=np.int32)
        first = np.empty(info["n_workers"], dtype=np.int32)
        _check(lib.gemm_get_log(self.h, owner.ctypes.data, claims.ctypes.data, first.ctypes.data,
                                info["n_tiles"], info["n_workers"]), "gemm_get_log")
        return owner, claims, first

    def get_trace(self):
        import numpy as np
        info = self.last_launch()
        out = np.empty((info["n_tiles"], 8), dtype=np.uint64)
        _check(lib.gemm_get_trace(self.h, out.ctypes.data, info["n_tiles"]), "gemm_get_trace")
        return out

    def max_active_clusters(self, tile=(128, 256, 64), cluster=1) -> int:
        n = ctypes.c_int()
        _check(lib.gemm_max_active_clusters(self.h, _tile(tile), _cluster(cluster), ctypes.byref(n)),
               "gemm_max_active_clusters")
        return n.value

    @property
    def sm_count(self) -> int:
        n = ctypes.c_int()
        _check(lib.gemm_sm_count(self.h, ctypes.byref(n)), "gemm_sm_count")
        return n.value

    def occupy_start(self, n_ctas: int, limit_ns: int = 20_000_000_000, stream=None) -> None:
        _check(lib.gemm_occupy_start(self.h, n_ctas, limit_ns, _stream(stream)), "gemm_occupy_start")

    def occupy_wait_resident(self, wait_ms: int = 5000) -> None:
        _check(lib.gemm_occupy_wait_resident(self.h, wait_ms), "gemm_occupy_wait_resident")

    def occupy_stop(self) -> int:
        st = ctypes.c_int()
        _check(lib.gemm_occupy_stop(self.h, ctypes.byref(st)), "gemm_occupy_stop")
        return st.value
