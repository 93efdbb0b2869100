"""Pins of the NVFP4 GEMM oracle ("Tensor Core" chapter, the table of tensor-core formats per
generation: Blackwell adds FP4 with block-scaled NVFP4 / MXFP4; read as E2M1 elements in
blocks of 16 along K sharing one UE4M3 scale, B given K-major).

E2M1 is checked on all 16 codes against the values its definition gives; UE4M3 on all
valid codes against torch's float8_e4m3fn; unit scales reduce the GEMM to numpy on the
decoded elements; a power of two per row / column scales it exactly; random block scales
with a K tail against numpy on scale-expanded operands (the scales vary along K, rows and
columns, so a misindexed scale fails); the packing (low nibble = even k) against a case
built by hand; a small case against exact rationals."""
import math
from fractions import Fraction

import numpy as np
import torch

import workloads as wl

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _unpack(P, cols):
    codes = np.empty((P.shape[0], 2 * P.shape[1]), np.uint8)
    codes[:, 0::2] = P & 15
    codes[:, 1::2] = P >> 4
    c = codes[:, :cols]
    mag = np.array(E2M1)[c & 7]
    return np.where(c & 8, -mag, mag)


def _ue4m3(S):
    return torch.from_numpy(np.ascontiguousarray(S)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e2m1_all_codes(orc):
    for c in range(16):
        want = E2M1[c & 7] * (-1.0 if c & 8 else 1.0)
        got = orc.decode_e2m1(c)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), c


def test_ue4m3_all_codes(orc):
    ref = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(127):
        assert orc.decode_ue4m3(c) == ref[c], c
    assert math.isnan(orc.decode_ue4m3(127))
    assert orc.decode_ue4m3(0x38) == 1.0 and orc.decode_ue4m3(126) == 448.0


def test_packing_low_nibble_is_even_k(orc):
    # A = [[1, 2]] packed as one byte: low nibble code of 1.0 (0x2), high nibble 2.0 (0x4)
    A = np.array([[0x42]], np.uint8)
    Bt = np.array([[0x22], [0x24]], np.uint8)  # column 0 = [1, 1], column 1 = [2, 1]
    one = np.full((2, 1), 0x38, np.uint8)
    D, _ = orc.gemm_nvf4(1, 2, 2, 1.0, A, 2, one[:1], 1, Bt, 2, one, 1)
    assert D.tolist() == [[3.0, 4.0]]


def test_unit_scales_against_numpy(orc):
    M, N, K = 20, 33, 96
    A, _ = wl.nvf4_quant(M, K, 1)
    Bt, _ = wl.nvf4_quant(N, K, 2)
    KB = K // 16
    ones_a = np.full((M, KB), 0x38, np.uint8)
    ones_b = np.full((N, KB), 0x38, np.uint8)
    D, _ = orc.gemm_nvf4(M, N, K, 1.0, A, K, ones_a, KB, Bt, K, ones_b, KB)
    np.testing.assert_allclose(D, _unpack(A, K) @ _unpack(Bt, K).T, rtol=0, atol=1e-12)


def test_power_of_two_scales_exact(orc):
    M, N, K = 8, 10, 64
    A, _ = wl.nvf4_quant(M, K, 3)
    Bt, _ = wl.nvf4_quant(N, K, 4)
    KB = K // 16
    one = lambda r: np.full((r, KB), 0x38, np.uint8)
    D1, _ = orc.gemm_nvf4(M, N, K, 1.0, A, K, one(M), KB, Bt, K, one(N), KB)
    t = np.arange(M) % 5 - 2
    u = np.arange(N) % 3 - 1
    SA = np.repeat(((t + 7) << 3).astype(np.uint8)[:, None], KB, axis=1)   # 2^t as UE4M3
    SB = np.repeat(((u + 7) << 3).astype(np.uint8)[:, None], KB, axis=1)
    D2, _ = orc.gemm_nvf4(M, N, K, 1.0, A, K, SA, KB, Bt, K, SB, KB)
    np.testing.assert_array_equal(D2, D1 * np.ldexp(1.0, t[:, None] + u[None, :]))


def test_random_scales_k_tail_against_numpy(orc):
    M, N, K, pad = 37, 45, 200, 8           # K not a multiple of 16
    A, SA = wl.nvf4_quant(M, K, 5, ld=K + pad)
    Bt, SB = wl.nvf4_quant(N, K, 6, ld=K + pad)
    KB = SA.shape[1]
    C = wl.f32_normal(M, N, 7)
    D, absab = orc.gemm_nvf4(M, N, K, 0.5, A, K + pad, SA, KB, Bt, K + pad, SB, KB, -2.0, C, N)
    kb = np.arange(K) // 16
    Ad = _unpack(A, K) * _ue4m3(SA)[:, kb]
    Bd = _unpack(Bt, K) * _ue4m3(SB)[:, kb]
    ref = 0.5 * Ad @ Bd.T - 2.0 * C.astype(np.float64)
    np.testing.assert_allclose(D, ref, rtol=0, atol=1e-12 * (1 + np.abs(Ad) @ np.abs(Bd).T).max())
    np.testing.assert_allclose(absab, np.abs(Ad) @ np.abs(Bd).T, rtol=1e-12)
    assert (SA != SA[:, :1]).any() and (SB != SB[:, :1]).any() and (SA != SA[:1]).any() and (SB != SB[:1]).any()


def test_small_case_exact_rationals(orc):
    M, N, K = 3, 2, 40
    A, SA = wl.nvf4_quant(M, K, 8)
    Bt, SB = wl.nvf4_quant(N, K, 9)
    KB = SA.shape[1]
    D, _ = orc.gemm_nvf4(M, N, K, 1.0, A, K, SA, KB, Bt, K, SB, KB)
    a, b, sa, sb = _unpack(A, K), _unpack(Bt, K), _ue4m3(SA), _ue4m3(SB)
    for i in range(M):
        for j in range(N):
            exact = sum(Fraction(a[i, k]) * Fraction(sa[i, k // 16]) * Fraction(b[j, k]) * Fraction(sb[j, k // 16])
                        for k in range(K))
            assert abs(Fraction(D[i, j]) - exact) <= abs(exact) * Fraction(1, 2 ** 50)
