"""Pins for the CPU oracle GEMM (no GPU).

Each test ties the oracle to something other than itself: the IEEE bfloat16
definition, exact rational arithmetic, closed forms, or numpy's integer matmul.
The set is chosen so that a dropped term, a wrong sign, a wrong index or a
transposed operand in the oracle fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle


def ieee_bf16_value(bits: int) -> Fraction:
    """bfloat16 = sign(1) | exponent(8, bias 127) | fraction(7), decoded with integers."""
    s = (bits >> 15) & 1
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    if e == 0xFF:
        raise ValueError("inf/nan")
    if e == 0:
        mag = Fraction(f, 128) * Fraction(2) ** -126
    else:
        mag = (1 + Fraction(f, 128)) * Fraction(2) ** (e - 127)
    return -mag if s else mag


def test_bf16_decode_known_patterns():
    cases = {0x3F80: 1.0, 0xBF80: -1.0, 0x4000: 2.0, 0xC040: -3.0, 0x3F81: 1.0078125,
             0x4049: 3.140625, 0x0000: 0.0, 0x8000: -0.0, 0x0001: 2.0 ** -133,
             0x7F7F: (2 - 2 ** -7) * 2.0 ** 127, 0x3E80: 0.25}
    got = oracle.bf16_decode(np.array(list(cases), dtype=np.uint16))
    assert list(got) == list(cases.values())


def test_bf16_decode_all_finite_patterns():
    bits = np.array([b for b in range(1 << 16) if ((b >> 7) & 0xFF) != 0xFF], dtype=np.uint16)
    got = oracle.bf16_decode(bits)
    for b, v in zip(bits[::97], got[::97]):
        assert Fraction(v) == ieee_bf16_value(int(b))


def _rand_bits(rng, shape, lo=-1.0, hi=1.0):
    import torch
    x = torch.from_numpy(rng.uniform(lo, hi, size=shape).astype(np.float32)).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (7, 3, 16), (13, 11, 9), (16, 16, 16), (5, 16, 2)])
def test_exact_rational_brute_force(M, N, K):
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    A = _rand_bits(rng, (M, K), -3, 3)
    B = _rand_bits(rng, (K, N), -3, 3)
    C = oracle.gemm(A, B)
    u = Fraction(1, 2 ** 53)
    gamma = (K - 1) * u / (1 - (K - 1) * u) if K > 1 else Fraction(0)
    for i in range(M):
        for j in range(N):
            terms = [ieee_bf16_value(int(A[i, k])) * ieee_bf16_value(int(B[k, j])) for k in range(K)]
            exact = sum(terms, Fraction(0))
            bound = gamma * sum(abs(t) for t in terms)
            assert abs(Fraction(C[i, j]) - exact) <= bound, (i, j)


def test_identity_gives_A():
    rng = np.random.default_rng(1)
    M, K, N = 9, 24, 40
    A = _rand_bits(rng, (M, K))
    one = 0x3F80
    B = np.zeros((K, N), dtype=np.uint16)
    B[np.arange(K), np.arange(K)] = one          # [I_K | 0]
    C = oracle.gemm(A, B)
    assert np.array_equal(C[:, :K], oracle.bf16_decode(A))
    assert np.all(C[:, K:] == 0.0)


def test_rank_one_closed_form():
    """Constant rows A[i][k] = u_i and B[k][j] = v_j give C = K * u_i * v_j exactly."""
    import torch
    M, N, K = 6, 10, 96
    u = np.array([1, -2, 0.5, 4, -0.25, 8], dtype=np.float32)
    v = np.array([1, 2, -1, 0.5, 0.125, -4, 16, -0.0625, 3, -6], dtype=np.float32)
    A = torch.from_numpy(np.repeat(u[:, None], K, axis=1)).to(torch.bfloat16)
    B = torch.from_numpy(np.repeat(v[None, :], K, axis=0)).to(torch.bfloat16)
    C = oracle.gemm(A, B)
    assert np.array_equal(C, K * np.outer(u.astype(np.float64), v.astype(np.float64)))


@pytest.mark.parametrize("M,N,K", [(37, 53, 71), (8, 16, 8192), (128, 64, 257)])
def test_integer_inputs_match_numpy_int64(M, N, K):
    import torch
    g = torch.Generator().manual_seed(M + N + K)
    a = torch.randint(-4, 5, (M, K), generator=g)
    b = torch.randint(-4, 5, (K, N), generator=g)
    C = oracle.gemm(a.to(torch.bfloat16), b.to(torch.bfloat16))
    ref = a.numpy().astype(np.int64) @ b.numpy().astype(np.int64)
    assert np.array_equal(C, ref.astype(np.float64))


def test_block_and_entries_match_full():
    rng = np.random.default_rng(7)
    M, N, K = 40, 33, 50
    A = _rand_bits(rng, (M, K))
    B = _rand_bits(rng, (K, N))
    C = oracle.gemm(A, B)
    assert np.array_equal(oracle.gemm_block(A, B, 3, 17, 5, 31), C[3:17, 5:31])
    rows = rng.integers(0, M, 50)
    cols = rng.integers(0, N, 50)
    assert np.array_equal(oracle.gemm_entries(A, B, rows, cols), C[rows, cols])


def test_tolerance_rule():
    ref = np.array([0.0, 10.0, -100.0])
    ok, _ = oracle.within_tolerance(ref + np.array([0.9e-3, 10.9e-3, -100.9e-3]), ref)
    assert ok
    ok, _ = oracle.within_tolerance(ref + np.array([0.0, 0.0, 0.2]), ref)
    assert not ok
    ok, _ = oracle.within_tolerance(np.array([np.nan, 10.0, -100.0]), ref)
    assert not ok


def test_planted_transpose_is_caught():
    """Reading B as N-major (a transposed operand) must fail the numpy pin."""
    import torch
    g = torch.Generator().manual_seed(3)
    a = torch.randint(-4, 5, (12, 12), generator=g)
    b = torch.randint(-4, 5, (12, 12), generator=g)
    wrong = oracle.gemm(a.to(torch.bfloat16), b.t().contiguous().to(torch.bfloat16))
    ref = a.numpy().astype(np.int64) @ b.numpy().astype(np.int64)
    assert not np.array_equal(wrong, ref.astype(np.float64))


def test_entries_against_exact_rationals():
    rng = np.random.default_rng(11)
    M, N, K = 9, 13, 11
    A = _rand_bits(rng, (M, K), -2, 2)
    B = _rand_bits(rng, (K, N), -2, 2)
    rows = rng.integers(0, M, 30)
    cols = rng.integers(0, N, 30)
    got = oracle.gemm_entries(A, B, rows, cols)
    u = Fraction(1, 2 ** 53)
    gamma = (K - 1) * u / (1 - (K - 1) * u)
    for e, (i, j) in enumerate(zip(rows, cols)):
        terms = [ieee_bf16_value(int(A[i, k])) * ieee_bf16_value(int(B[k, j])) for k in range(K)]
        assert abs(Fraction(got[e]) - sum(terms, Fraction(0))) <= gamma * sum(abs(t) for t in terms)


def test_block_against_numpy_int64():
    import torch
    g = torch.Generator().manual_seed(12)
    a = torch.randint(-4, 5, (70, 300), generator=g)
    b = torch.randint(-4, 5, (300, 90), generator=g)
    blk = oracle.gemm_block(a.to(torch.bfloat16), b.to(torch.bfloat16), 17, 61, 5, 83)
    ref = a.numpy().astype(np.int64)[17:61] @ b.numpy().astype(np.int64)[:, 5:83]
    assert np.array_equal(blk, ref.astype(np.float64))


def test_transpose_identity_bit_exact():
    """(A B)^T = B^T A^T: both sides sum the same exact products in ascending k, so the
    oracle must return the transpose bit for bit (an i/j index swap anywhere breaks it)."""
    import torch
    rng = np.random.default_rng(21)
    A = _rand_bits(rng, (37, 29))
    B = _rand_bits(rng, (29, 45))
    C = oracle.gemm(A, B)
    At = torch.from_numpy(A.view(np.int16)).t().contiguous().view(torch.bfloat16)
    Bt = torch.from_numpy(B.view(np.int16)).t().contiguous().view(torch.bfloat16)
    assert np.array_equal(oracle.gemm(Bt, At), C.T)


def test_depth_scaled_tolerance_rule():
    """The acceptance rule for products deeper than the stated workloads: the stated 1e-3
    up to K = 8192, then scaled by (K / 8192)^1.5 (the growth of the tensor cores'
    accumulation error bound); monotone, and exactly the stated value at the stated depths."""
    from tests.gpu_helpers import rel_tolerance
    assert rel_tolerance(0) == rel_tolerance(1000) == rel_tolerance(8192) == 1e-3
    assert abs(rel_tolerance(16384) - 1e-3 * 2 ** 1.5) < 1e-15
    assert abs(rel_tolerance(12800) - 1e-3 * (12800 / 8192) ** 1.5) < 1e-15
    ks = [8192, 9000, 10752, 12544, 12800, 16384]
    assert all(rel_tolerance(a) < rel_tolerance(b) for a, b in zip(ks, ks[1:]))
