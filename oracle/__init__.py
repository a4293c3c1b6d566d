"""CPU oracle: the plain GEMM (binary64 accumulation over bf16 inputs) and the
tile-coverage model of the scheduling policies.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  The
product library never calls it and there is no CPU fallback built on it.

The GEMM lives in ``gemm_ref.c`` (compiled by ``oracle/build.py`` into
``liboracle.so``); this module only marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import coverage  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        from .build import build
        build()
    lib = ctypes.CDLL(LIB_PATH)
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_gemm.argtypes = [i64, i64, i64, p, p, p]
    lib.oracle_gemm.restype = None
    lib.oracle_gemm_block.argtypes = [i64, i64, i64, p, p, i64, i64, i64, i64, p]
    lib.oracle_gemm_block.restype = None
    lib.oracle_gemm_entries.argtypes = [i64, i64, i64, p, p, i64, p, p, p]
    lib.oracle_gemm_entries.restype = None
    lib.oracle_bf16_decode.argtypes = [i64, p, p]
    lib.oracle_bf16_decode.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    _lib = lib
    return lib


def _bits(x) -> np.ndarray:
    """Accept a uint16 numpy array of bf16 bit patterns or a torch bfloat16 tensor."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("expected bf16 bit patterns as uint16")
        return np.ascontiguousarray(x)
    try:
        import torch
    except ImportError as e:  # pragma: no cover
        raise TypeError("unsupported input") from e
    if isinstance(x, torch.Tensor):
        if x.dtype != torch.bfloat16:
            raise TypeError("expected a bfloat16 tensor")
        return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    raise TypeError("unsupported input")


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def bf16_decode(bits) -> np.ndarray:
    b = _bits(np.asarray(bits, dtype=np.uint16))
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_bf16_decode(b.size, _ptr(b), _ptr(out))
    return out


def gemm(A, B) -> np.ndarray:
    """C = A @ B in binary64; A is M x K, B is K x N (bf16)."""
    a, b = _bits(A), _bits(B)
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    out = np.empty((M, N), dtype=np.float64)
    _load().oracle_gemm(M, N, K, _ptr(a), _ptr(b), _ptr(out))
    return out


def gemm_block(A, B, r0: int, r1: int, c0: int, c1: int) -> np.ndarray:
    """Rows [r0, r1) and columns [c0, c1) of A @ B in binary64."""
    a, b = _bits(A), _bits(B)
    M, K = a.shape
    K2, N = b.shape
    if K != K2 or not (0 <= r0 <= r1 <= M and 0 <= c0 <= c1 <= N):
        raise ValueError("bad block")
    out = np.empty((r1 - r0, c1 - c0), dtype=np.float64)
    _load().oracle_gemm_block(M, N, K, _ptr(a), _ptr(b), r0, r1, c0, c1, _ptr(out))
    return out


def gemm_entries(A, B, rows, cols) -> np.ndarray:
    """Single elements (rows[e], cols[e]) of A @ B in binary64."""
    a, b = _bits(A), _bits(B)
    M, K = a.shape
    K2, N = b.shape
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if K != K2 or r.shape != c.shape or (r.size and (r.min() < 0 or r.max() >= M or c.min() < 0 or c.max() >= N)):
        raise ValueError("bad entries")
    out = np.empty(r.shape, dtype=np.float64)
    _load().oracle_gemm_entries(M, N, K, _ptr(a), _ptr(b), r.size, _ptr(r), _ptr(c), _ptr(out))
    return out


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def within_tolerance(c_gpu: np.ndarray, c_ref: np.ndarray, rel: float = 1e-3):
    """Elementwise acceptance |C_gpu - C_ref| <= rel * (1 + |C_ref|); returns
    (ok, worst ratio of error to allowance)."""
    c_gpu = np.asarray(c_gpu, dtype=np.float64)
    err = np.abs(c_gpu - c_ref)
    allow = rel * (1.0 + np.abs(c_ref))
    ratio = float(np.max(err / allow)) if err.size else 0.0
    ok = bool(np.all(np.isfinite(c_gpu))) and ratio <= 1.0
    return ok, ratio
