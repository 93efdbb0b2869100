"""Pins of the MX block-scaled GEMM oracle ("Tensor Core" chapter, the table of tensor-core
formats per generation: Blackwell adds block-scaled formats such as MXFP4 / NVFP4; read
as OCP microscaling: one E8M0 scale 2^(e-127) per 32 consecutive K elements of a row of A
or a column of B).

Scales are stored K-block-contiguous: SA[i][kb] per row of A, SB[j][kb] per column of B.
The E8M0 decoder is checked on all 256 codes against ldexp; unit scales reduce the GEMM
to the plain 8-bit GEMM (checked against the separate block-scaled oracle function with
unit FP32 scales, and against numpy on torch-decoded codes); a power of two per row and
column scales the result exactly; random block scales with ragged K and N tails are
checked against numpy matmul of operands expanded by the scales (so a transposed or
misindexed scale fails); a small case is checked against exact rationals.
"""
import math
from fractions import Fraction

import numpy as np
import torch

import workloads as wl


def _dec(bits, fmt):
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    return torch.from_numpy(np.ascontiguousarray(bits)).view(dt).to(torch.float64).numpy()


def _scaled(A, SA, B, SB, M, N, K, a_fmt, b_fmt):
    """Operands with their block scales applied, from torch's decoders and numpy."""
    kb = np.arange(K) // 32
    Ad = _dec(A[:, :K], a_fmt) * np.ldexp(1.0, SA[:, kb].astype(np.int64) - 127)
    Bd = _dec(B[:, :N], b_fmt) * np.ldexp(1.0, SB[:N, kb].T.astype(np.int64) - 127)
    return Ad, Bd


def test_ue8m0_decoder_all_codes(orc):
    for e in range(255):
        assert orc.decode_ue8m0(e) == math.ldexp(1.0, e - 127), e
    assert math.isnan(orc.decode_ue8m0(255))
    assert orc.decode_ue8m0(127) == 1.0
    assert orc.decode_ue8m0(0) == 2.0 ** -127


def test_unit_scales_reduce_to_the_plain_8bit_gemm(orc):
    M, N, K = 23, 70, 150
    for a_fmt, b_fmt in [("e4m3", "e4m3"), ("e5m2", "e4m3"), ("e4m3", "e5m2")]:
        A, _ = wl.mx_quant(M, K, 11, 1, fmt=a_fmt)
        B, _ = wl.mx_quant(K, N, 12, 0, fmt=b_fmt)
        KB = -(-K // 32)
        SA = np.full((M, KB), 127, np.uint8)
        SB = np.full((N, KB), 127, np.uint8)
        D, _ = orc.gemm_mx_f8(a_fmt, b_fmt, M, N, K, 1.0, A.ravel(), K, SA.ravel(), KB, B.ravel(), N,
                              SB.ravel(), KB)
        # the separate FP8 block-scaled oracle function with unit FP32 scales
        kb128, nb128 = -(-K // 128), -(-N // 128)
        D2, _ = orc.gemm_f8_blockscaled_mixed(a_fmt, b_fmt, M, N, K, 1.0, A.ravel(), K,
                                              np.ones((M, kb128), np.float32).ravel(), kb128, B.ravel(), N,
                                              np.ones((kb128, nb128), np.float32).ravel(), nb128)
        np.testing.assert_array_equal(D, D2)
        ref = _dec(A, a_fmt) @ _dec(B, b_fmt)
        np.testing.assert_allclose(D, ref, rtol=1e-12, atol=1e-12)


def test_power_of_two_row_and_column_scales_are_exact(orc):
    M, N, K = 9, 40, 96
    A, _ = wl.mx_quant(M, K, 21, 1)
    B, _ = wl.mx_quant(K, N, 22, 0)
    KB = K // 32
    ones_a = np.full((M, KB), 127, np.uint8)
    ones_b = np.full((N, KB), 127, np.uint8)
    D1, _ = orc.gemm_mx_f8("e4m3", "e4m3", M, N, K, 1.0, A.ravel(), K, ones_a.ravel(), KB, B.ravel(), N,
                           ones_b.ravel(), KB)
    t = np.arange(M) % 7 - 3          # 2^t per row of A (same for every K block)
    u = np.arange(N) % 5 - 2          # 2^u per column of B
    SA = np.repeat((127 + t)[:, None], KB, axis=1).astype(np.uint8)
    SB = np.repeat((127 + u)[:, None], KB, axis=1).astype(np.uint8)
    D2, _ = orc.gemm_mx_f8("e4m3", "e4m3", M, N, K, 1.0, A.ravel(), K, SA.ravel(), KB, B.ravel(), N,
                           SB.ravel(), KB)
    np.testing.assert_array_equal(D2, D1 * np.ldexp(1.0, t[:, None] + u[None, :]))


def test_random_block_scales_ragged_tails_against_numpy(orc):
    for (M, N, K, pad, a_fmt, b_fmt, seed) in [(37, 133, 200, 5, "e4m3", "e4m3", 31),
                                               (64, 64, 32, 0, "e5m2", "e5m2", 32),
                                               (5, 300, 77, 3, "e4m3", "e5m2", 33)]:
        A, SA = wl.mx_quant(M, K, seed, 1, ld=K + pad, fmt=a_fmt)
        B, SB = wl.mx_quant(K, N, seed + 100, 0, ld=N + pad, fmt=b_fmt)
        KB = SA.shape[1]
        # pad the scale matrices too, with codes that would be wrong if read
        SAp = np.full((M, KB + 2), 200, np.uint8)
        SAp[:, :KB] = SA
        SBp = np.full((N, KB + 3), 200, np.uint8)
        SBp[:, :KB] = SB
        C = wl.f32_normal(M, N, seed + 200)
        D, absab = orc.gemm_mx_f8(a_fmt, b_fmt, M, N, K, 0.75, A.ravel(), K + pad, SAp.ravel(), KB + 2,
                                  B.ravel(), N + pad, SBp.ravel(), KB + 3, -1.5, C.ravel(), N)
        Ad, Bd = _scaled(A, SA, B, SB, M, N, K, a_fmt, b_fmt)
        ref = 0.75 * (Ad @ Bd) - 1.5 * C.astype(np.float64)
        scale = np.abs(Ad) @ np.abs(Bd)
        np.testing.assert_allclose(D, ref, rtol=0, atol=1e-12 * (1 + np.max(scale)))
        np.testing.assert_allclose(absab, scale, rtol=1e-12)
        # the scales vary along K and across rows / columns, so a scale taken from the wrong
        # block, row or column would change the result
        if KB > 1:
            assert (SA != SA[:, :1]).any() and (SB != SB[:, :1]).any()
        assert (SA != SA[:1, :]).any() and (SB != SB[:1, :]).any()


def test_small_case_exact_rationals(orc):
    M, N, K = 3, 4, 70                  # three K blocks, the last one 6 long
    A, SA = wl.mx_quant(M, K, 41, 1)
    B, SB = wl.mx_quant(K, N, 42, 0)
    KB = SA.shape[1]
    D, _ = orc.gemm_mx_f8("e4m3", "e4m3", M, N, K, 1.0, A.ravel(), K, SA.ravel(), KB, B.ravel(), N,
                          SB.ravel(), KB)
    Ad = _dec(A, "e4m3")
    Bd = _dec(B, "e4m3")
    for i in range(M):
        for j in range(N):
            exact = sum(Fraction(Ad[i, k]) * Fraction(2) ** (int(SA[i, k // 32]) - 127) *
                        Fraction(Bd[k, j]) * Fraction(2) ** (int(SB[j, k // 32]) - 127) for k in range(K))
            assert abs(Fraction(D[i, j]) - exact) <= abs(exact) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200)


def test_generator_follows_the_mx_rule():
    """Input generator check: each block's largest scaled magnitude lies in [2^emax, 2^(emax+1))
    times its scale, and no element exceeds the format's maximum."""
    A, SA = wl.mx_quant(16, 96, 51, 1)
    Ad = _dec(A, "e4m3")
    for b in range(3):
        blk = np.abs(Ad[:, 32 * b:32 * b + 32]).max(axis=1)
        assert np.all(blk <= 448.0)
        assert np.all(blk >= 2.0 ** 7)  # amax / 2^X >= 2^8 before rounding, >= 2^7 after saturating rounding
