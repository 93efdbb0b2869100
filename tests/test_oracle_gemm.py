"""Pins of the GEMM oracle, D = alpha * A x B + beta * C ("Tensor Core" chapter,
section "Tensor Core 做什么"; alpha/beta generalisation as in the BLAS reading).

Nothing here re-types the oracle's formula: every check compares it with an
independent fact -- an exact rational brute force, a closed form (identity or
permutation B, all-ones A, rank-1 operands, small integers), a library routine
(numpy float64 matmul), or linearity -- with non-square shapes and padded leading
dimensions so that a transposed operand or a wrong index fails.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads as wl


def _dec(kind, bits):
    if kind == "f16":
        return bits.view(np.float16).astype(np.float64)
    if kind == "bf16":
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    if kind == "e4m3":
        return torch.from_numpy(bits.view(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    raise ValueError(kind)


def _f16_bits(vals):
    return np.asarray(vals, dtype=np.float64).astype(np.float16).view(np.uint16)


def _bf16_bits(vals):
    t = torch.tensor(np.asarray(vals, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (4, 4, 4), (3, 5, 1), (2, 3, 7)])
def test_bruteforce_exact_rationals(orc, M, N, K):
    A = wl.f16_uniform(M, K, 21)
    B = wl.f16_uniform(K, N, 22)
    C = wl.f32_normal(M, N, 23)
    alpha, beta = 0.75, -1.5
    D, S = orc.gemm("f16", M, N, K, alpha, A.ravel(), K, B.ravel(), N, beta, C.ravel(), N)
    a = [[Fraction(float(v)) for v in row] for row in A.view(np.float16).astype(np.float64)]
    b = [[Fraction(float(v)) for v in row] for row in B.view(np.float16).astype(np.float64)]
    for i in range(M):
        for j in range(N):
            exact = Fraction(alpha) * sum(a[i][k] * b[k][j] for k in range(K)) + \
                Fraction(beta) * Fraction(float(C[i, j]))
            sabs = sum(abs(a[i][k] * b[k][j]) for k in range(K))
            assert abs(Fraction(D[i, j]) - exact) <= Fraction(2.0 ** -50) * (sabs + abs(Fraction(float(C[i, j]))) + 1)
            assert abs(Fraction(S[i, j]) - sabs) <= Fraction(2.0 ** -50) * sabs


@pytest.mark.parametrize("kind", ["f16", "bf16"])
def test_identity_B(orc, kind):
    M, K = 7, 9
    A = wl.operand(kind, M, K, 31, ld=12)
    eye = np.eye(K)
    B = _f16_bits(eye) if kind == "f16" else _bf16_bits(eye)
    C = wl.f32_normal(M, K, 33, ld=10)
    alpha, beta = 1.25, 0.5
    D, _ = orc.gemm(kind, M, K, K, alpha, A.ravel(), 12, B.ravel(), K, beta, C.ravel(), 10)
    want = alpha * _dec(kind, A[:, :K]) + beta * C[:, :K].astype(np.float64)
    assert np.array_equal(D, want)


def test_permutation_B(orc):
    M, K = 6, 8
    A = wl.f16_uniform(M, K, 41)
    perm = np.random.default_rng(42).permutation(K)
    P = np.zeros((K, K))
    P[perm, np.arange(K)] = 1.0  # column j of A x P is column perm[j] of A
    D, _ = orc.gemm("f16", M, K, K, 1.0, A.ravel(), K, _f16_bits(P).ravel(), K)
    assert np.array_equal(D, _dec("f16", A)[:, perm])


def test_all_ones_A_gives_column_sums(orc):
    M, N, K = 3, 11, 256
    A = _f16_bits(np.ones((M, K)))
    B = wl.f16_uniform(K, N, 51)
    D, _ = orc.gemm("f16", M, N, K, 1.0, A.ravel(), K, B.ravel(), N)
    Bd = _dec("f16", B)
    # each column sum is a multiple of 2^-24 below 2^9: exact in double; compare with exact rationals
    for j in range(N):
        exact = sum(Fraction(float(v)) for v in Bd[:, j])
        assert all(Fraction(D[i, j]) == exact for i in range(M))


def test_rank_one(orc):
    M, N, K = 5, 6, 13
    u = np.random.default_rng(61).uniform(-1, 1, M).astype(np.float16).astype(np.float64)
    v = np.random.default_rng(62).uniform(-1, 1, N).astype(np.float16).astype(np.float64)
    A = _f16_bits(np.repeat(u[:, None], K, axis=1))   # A = u 1^T
    Bv = np.zeros((K, N))
    Bv[0] = v                                         # B = e_0 v^T
    C = wl.f32_normal(M, N, 63)
    D, _ = orc.gemm("f16", M, N, K, 2.0, A.ravel(), K, _f16_bits(Bv).ravel(), N, -0.5, C.ravel(), N)
    assert np.array_equal(D, 2.0 * np.outer(u, v) + (-0.5) * C.astype(np.float64))


def test_linearity_alpha_beta(orc):
    M, N, K = 9, 7, 33
    A = wl.bf16_normal(M, K, 71)
    B = wl.bf16_normal(K, N, 72)
    C = wl.f32_normal(M, N, 73)
    D10, _ = orc.gemm("bf16", M, N, K, 1.0, A.ravel(), K, B.ravel(), N)
    for alpha, beta in [(0.5, -1.25), (3.0, 2.0), (-1.0, 0.0)]:
        D, _ = orc.gemm("bf16", M, N, K, alpha, A.ravel(), K, B.ravel(), N, beta, C.ravel(), N)
        want = alpha * D10 + beta * C.astype(np.float64)
        assert np.allclose(D, want, rtol=4e-16, atol=1e-300 + 4e-16 * np.abs(want).max())


def test_small_integers_exact(orc):
    rng = np.random.default_rng(81)
    M, N, K = 10, 12, 64
    Ai = rng.integers(-8, 9, size=(M, K))
    Bi = rng.integers(-8, 9, size=(K, N))
    D, S = orc.gemm("f16", M, N, K, 1.0, _f16_bits(Ai).ravel(), K, _f16_bits(Bi).ravel(), N)
    assert np.array_equal(D, (Ai.astype(np.int64) @ Bi.astype(np.int64)).astype(np.float64))
    assert np.array_equal(S, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64))


@pytest.mark.parametrize("kind", ["f16", "bf16", "e4m3"])
def test_numpy_matmul_crosscheck(orc, kind):
    M, N, K, lda, ldb = 37, 29, 71, 80, 40
    if kind == "e4m3":
        A = wl.e4m3_blockquant(M, K, 91, 1, 1 << 20, ld=lda)[0]
        B = wl.e4m3_blockquant(K, N, 92, 1 << 20, 1, ld=ldb)[0]
    else:
        A = wl.operand(kind, M, K, 91, ld=lda)
        B = wl.operand(kind, K, N, 92, ld=ldb)
    C = wl.f32_normal(M, N, 93, ld=33)
    D, S = orc.gemm(kind, M, N, K, 0.5, A.ravel(), lda, B.ravel(), ldb, -1.25, C.ravel(), 33)
    Ad, Bd = _dec(kind, A[:, :K]), _dec(kind, B[:, :N])
    want = 0.5 * (Ad @ Bd) + (-1.25) * C[:, :N].astype(np.float64)
    sab = np.abs(Ad) @ np.abs(Bd)
    assert np.all(np.abs(D - want) <= 1e-13 * (sab + np.abs(C[:, :N])) + 1e-300)
    assert np.allclose(S, sab, rtol=1e-13, atol=0)


def test_selected_rows_match_full(orc):
    M, N, K = 20, 9, 17
    A = wl.f16_uniform(M, K, 101)
    B = wl.f16_uniform(K, N, 102)
    Dfull, _ = orc.gemm("f16", M, N, K, 1.0, A.ravel(), K, B.ravel(), N)
    rows = [19, 0, 7]
    Dsel, _ = orc.gemm("f16", M, N, K, 1.0, A.ravel(), K, B.ravel(), N, rows=rows)
    assert np.array_equal(Dsel, Dfull[rows])


def test_beta_zero_does_not_read_C(orc):
    M, N, K = 4, 4, 4
    A = wl.f16_uniform(M, K, 111)
    B = wl.f16_uniform(K, N, 112)
    C = np.full((M, N), np.nan, dtype=np.float32)
    D, _ = orc.gemm("f16", M, N, K, 1.0, A.ravel(), K, B.ravel(), N, 0.0, C.ravel(), N)
    assert np.all(np.isfinite(D))


def test_k_zero_gives_beta_C(orc):
    M, N = 3, 5
    C = wl.f32_normal(M, N, 121)
    D, _ = orc.gemm("f16", M, N, 0, 1.0, np.zeros(1, np.uint16), 1, np.zeros(1, np.uint16), N,
                    -1.25, C.ravel(), N)
    assert np.array_equal(D, -1.25 * C.astype(np.float64))
