"""Pins of the FP8 block-scaled GEMM oracle and the W8A8 GEMV oracle.

FP8 ("Tensor Core" chapter, "精度" section: FP8 needs scaling factors per tensor,
row or block): unit scales reduce it to a plain E4M3 GEMM, checked against numpy
matmul of torch-decoded codes; power-of-two and random block scales are checked
against numpy matmul of the scaled, expanded operands, with ragged K and N tails
so a wrong block index (j % 128 for j / 128, a transposed scale matrix) fails.

W8A8 ("NVIDIA A100: chip to SIMT", sections 5.1, 5.2): one-hot and all-ones
activations, the extreme codes, the INT32 bound printed in section 5.1, numpy int64
matmul, and the FP32 dequantisation sequence checked against numpy float32.
"""
import os

import numpy as np
import pytest
import torch

import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    return vals


def _e4m3(bits):
    return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _expand(sA, sB, M, N, K):
    """Per-element scale maps: sA over (i, k) from 1x128 blocks, sB over (k, j) from 128x128."""
    kb = np.arange(K) // 128
    SA = sA[:, kb].astype(np.float64)                       # M x K
    SB = sB[kb][:, np.arange(N) // 128].astype(np.float64)  # K x N
    return SA, SB


def _fp8_case(M, N, K, seed, ld_pad=0):
    A, sA = wl.e4m3_blockquant_rowblocks(M, K, seed, ld=K + ld_pad)
    B, sB = wl.e4m3_blockquant(K, N, seed + 1, 128, 128, ld=N + ld_pad)
    return A, sA, B, sB


def test_fp8_unit_scales_is_plain_e4m3(orc):
    M, N, K = 19, 150, 300
    A, _, B, _ = _fp8_case(M, N, K, 201)
    KB, NB = -(-K // 128), -(-N // 128)
    ones_a = np.ones((M, KB), np.float32)
    ones_b = np.ones((KB, NB), np.float32)
    D, _ = orc.gemm_fp8_blockscaled(M, N, K, 1.0, A.ravel(), K, ones_a.ravel(), KB, B.ravel(), N,
                                    ones_b.ravel(), NB)
    Ad, Bd = _e4m3(A), _e4m3(B)
    want = Ad @ Bd
    assert np.all(np.abs(D - want) <= 1e-13 * (np.abs(Ad) @ np.abs(Bd)))


def test_fp8_power_of_two_scales_exact_factor(orc):
    M, N, K = 5, 130, 256
    A, _, B, _ = _fp8_case(M, N, K, 211)
    # one scale 2^e for everything: the result is exactly 2^e times the unscaled one
    KB, NB = 2, 2
    D1, _ = orc.gemm_fp8_blockscaled(M, N, K, 1.0, A.ravel(), K, np.ones(M * KB, np.float32), KB,
                                     B.ravel(), N, np.ones(KB * NB, np.float32), NB)
    sa = np.full((M, KB), 2.0 ** -3, np.float32)
    sb = np.full((KB, NB), 2.0 ** 5, np.float32)
    D4, _ = orc.gemm_fp8_blockscaled(M, N, K, 1.0, A.ravel(), K, sa.ravel(), KB, B.ravel(), N,
                                     sb.ravel(), NB)
    assert np.array_equal(D4, D1 * 4.0)


@pytest.mark.parametrize("M,N,K,pad", [(7, 300, 389, 0), (16, 128, 128, 16), (3, 129, 1, 0)])
def test_fp8_random_scales_vs_numpy(orc, M, N, K, pad):
    A, sA, B, sB = _fp8_case(M, N, K, 221 + K, ld_pad=pad)
    KB, NB = sA.shape[1], sB.shape[1]
    C = wl.f32_normal(M, N, 225)
    D, S = orc.gemm_fp8_blockscaled(M, N, K, 0.5, A.ravel(), K + pad, sA.ravel(), KB, B.ravel(),
                                    N + pad, sB.ravel(), NB, -1.25, C.ravel(), N)
    SA, SB = _expand(sA, sB, M, N, K)
    Ad = _e4m3(A[:, :K]) * SA
    Bd = _e4m3(B[:, :N]) * SB
    want = 0.5 * (Ad @ Bd) - 1.25 * C.astype(np.float64)
    sab = np.abs(Ad) @ np.abs(Bd)
    assert np.all(np.abs(D - want) <= 1e-12 * (sab + np.abs(C)) + 1e-300)
    assert np.allclose(S, sab, rtol=1e-12, atol=0)


def test_fp8_scale_index_mistakes_would_be_caught(orc):
    """Non-uniform sB makes j//128 vs j%128 and sB vs sB^T give different answers."""
    M, N, K = 4, 256, 256
    A, sA, B, sB = _fp8_case(M, N, K, 231)
    sB = np.array([[1.0, 8.0], [0.25, 2.0]], np.float32)  # asymmetric on purpose
    D, _ = orc.gemm_fp8_blockscaled(M, N, K, 1.0, A.ravel(), K, sA.ravel(), 2, B.ravel(), N,
                                    sB.ravel(), 2)
    SA, SB = _expand(sA, sB, M, N, K)
    good = (_e4m3(A) * SA) @ (_e4m3(B) * SB)
    SBt = _expand(sA, sB.T.copy(), M, N, K)[1]
    wrong = (_e4m3(A) * SA) @ (_e4m3(B) * SBt)
    assert np.allclose(D, good, rtol=1e-12, atol=1e-12)
    assert not np.allclose(D, wrong, rtol=1e-3, atol=1e-3)


# ------------------------------------------------------------------ W8A8


def test_gemv_one_hot_and_all_ones(orc):
    N, K = 33, 96
    W = wl.int8_uniform((N, K), 301)
    sW = wl.scales_uniform(N, 302)
    for k in [0, 5, K - 1]:
        x = np.zeros(K, np.int8)
        x[k] = 1
        z, _ = orc.gemv_w8a8(N, K, x, 0.01, W, K, sW)
        assert np.array_equal(z, W[:, k].astype(np.int64))
    z, _ = orc.gemv_w8a8(N, K, np.ones(K, np.int8), 0.01, W, K, sW)
    assert np.array_equal(z, W.astype(np.int64).sum(axis=1))


def test_gemv_printed_int32_bound(orc):
    g = _golden("w8a8_int32_bound.txt")
    K = g["K"]
    q = -g["q_abs_max"]  # -128 is the one int8 code with |q| = 128
    x = np.full(K, q, np.int8)
    W = np.full((2, K), q, np.int8)
    W[1] = -q - 1  # 127
    z, _ = orc.gemv_w8a8(2, K, x, 1.0, W, K, np.ones(2, np.float32))
    assert z[0] == g["z_bound"] == K * 128 * 128
    assert z[0] < g["int32_limit"] == 2 ** 31
    assert z[1] == -K * 128 * 127


def test_gemv_extremes_of_generated_range(orc):
    K = 4096
    x = np.full(K, 127, np.int8)
    W = np.stack([np.full(K, 127, np.int8), np.full(K, -127, np.int8)])
    z, y = orc.gemv_w8a8(2, K, x, 0.02, W, K, np.full(2, 0.02, np.float32))
    assert list(z) == [66064384, -66064384]
    # float(66064384) is exact (66064384 = 2^10 * 64516), then two FP32 products
    want = ((np.float32(66064384) * np.float32(0.02)) * np.float32(0.02)).astype(np.float16)
    assert y[0] == want and y[1] == -want


def test_gemv_overflow_detected(orc):
    K = 140000  # 140000 * 127^2 > 2^31
    x = np.full(K, 127, np.int8)
    W = np.full((1, K), 127, np.int8)
    with pytest.raises(OverflowError):
        orc.gemv_w8a8(1, K, x, 1.0, W, K, np.ones(1, np.float32))


@pytest.mark.parametrize("N,K,ldw", [(11, 4096, 4096), (64, 100, 112), (5, 1, 16)])
def test_gemv_vs_numpy(orc, N, K, ldw):
    x, sx, W, sW = wl.int8_uniform(K, 311), np.float32(0.0137), None, wl.scales_uniform(N, 312)
    Wv = wl.int8_uniform((N, K), 313)
    W = np.full((N, ldw), 77, np.int8)
    W[:, :K] = Wv
    z, y = orc.gemv_w8a8(N, K, x, sx, W, ldw, sW)
    zn = Wv.astype(np.int64) @ x.astype(np.int64)
    assert np.array_equal(z, zn)
    # the dequantisation sequence in numpy float32: float(z), * s_x, * s_W[o], then to FP16
    yn = ((zn.astype(np.float32) * np.float32(sx)) * sW).astype(np.float16)
    assert np.array_equal(y.view(np.uint16), yn.view(np.uint16))
    # and within one FP16 ulp of the exact double-precision dequantisation
    exact = zn.astype(np.float64) * float(sx) * sW.astype(np.float64)
    ulp = np.spacing(np.abs(exact).astype(np.float16)).astype(np.float64)
    assert np.all(np.abs(y.astype(np.float64) - exact) <= ulp)


def test_gemv_large_z_rounds_through_float(orc):
    # |z| > 2^24 is not exactly representable in FP32: float(z) rounds first
    K = 2048
    x = np.full(K, 127, np.int8)
    W = np.full((1, K), 127, np.int8)
    W[0, 0] = 126  # z = 2048*127^2 - 127 = 33032065 (odd, > 2^24)
    z, y = orc.gemv_w8a8(1, K, x, 2.0 ** -10, W, K, np.full(1, 2.0 ** -10, np.float32))
    assert z[0] == 33032065
    assert int(np.float32(33032065)) == 33032064  # the int -> FP32 rounding step is real
    want = ((np.float32(33032064) * np.float32(2.0 ** -10)) * np.float32(2.0 ** -10)).astype(np.float16)
    assert y[0] == want


def test_generated_gemv_workload_fits_int32(orc):
    x, sx, W, sW = wl.gemv_inputs(256, 4096)
    z, y = orc.gemv_w8a8(256, 4096, x, sx, W, 4096, sW)
    assert np.all(np.abs(z) <= 4096 * 127 * 127)
    assert np.all(np.isfinite(y.astype(np.float32)))


def _f8(bits, fmt):
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    return torch.from_numpy(np.ascontiguousarray(bits)).view(dt).to(torch.float64).numpy()


@pytest.mark.parametrize("a_fmt,b_fmt", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
def test_f8_mixed_formats_vs_numpy(orc, a_fmt, b_fmt):
    M, N, K = 9, 260, 300
    A, sA = wl.e4m3_blockquant_rowblocks(M, K, 241, fmt=a_fmt)
    B, sB = wl.e4m3_blockquant(K, N, 242, 128, 128, fmt=b_fmt)
    KB, NB = sA.shape[1], sB.shape[1]
    D, S = orc.gemm_f8_blockscaled_mixed(a_fmt, b_fmt, M, N, K, 1.0, A.ravel(), K, sA.ravel(), KB,
                                         B.ravel(), N, sB.ravel(), NB)
    SA, SB = _expand(sA, sB, M, N, K)
    Ad = _f8(A, a_fmt) * SA
    Bd = _f8(B, b_fmt) * SB
    assert np.all(np.abs(D - Ad @ Bd) <= 1e-12 * (np.abs(Ad) @ np.abs(Bd)) + 1e-300)


def test_f8_mixed_e4m3_pair_equals_fp8_entry(orc):
    M, N, K = 5, 130, 200
    A, sA, B, sB = _fp8_case(M, N, K, 251)
    KB, NB = sA.shape[1], sB.shape[1]
    D1, _ = orc.gemm_fp8_blockscaled(M, N, K, 1.0, A.ravel(), K, sA.ravel(), KB, B.ravel(), N,
                                     sB.ravel(), NB)
    D2, _ = orc.gemm_f8_blockscaled_mixed("e4m3", "e4m3", M, N, K, 1.0, A.ravel(), K, sA.ravel(), KB,
                                          B.ravel(), N, sB.ravel(), NB)
    assert np.array_equal(D1, D2)
