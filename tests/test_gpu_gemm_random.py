"""Randomised GPU parity sweep of the GEMM entry points against the CPU oracle (seeded,
so every run checks the same cases): FP16 / BF16 / FP8 E4M3 and E5M2 operands, random
sizes from a few rows to several CTA-pair tiles, padded and TMA-illegal pitches,
alpha / beta, every output type, the allocation-free entry.  Every element is compared,
at the tolerance bar of the other GEMM tests, and D must have been written in full."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import assert_fully_written, check_all_rows, out_code, out_tensor, up

pytestmark = pytest.mark.gpu

OUTS = ["f32", "bf16", "f16"]


def _case(seed):
    rng = np.random.default_rng(9000 + seed)
    big = rng.random() < 0.3  # some cases large enough for the CTA-pair kernel
    M = int(rng.integers(300, 1500) if big else rng.integers(1, 400))
    N = int(rng.integers(300, 1500) if big else rng.integers(1, 400))
    K = int(rng.integers(1, 1200))
    pad_a = int(rng.choice([0, 0, 8, 16, 3]))
    pad_b = int(rng.choice([0, 0, 8, 32, 5]))
    alpha = float(rng.choice([1.0, 0.5, -2.0]))
    beta = float(rng.choice([0.0, 0.0, 1.0, -0.75]))
    out = OUTS[int(rng.integers(0, 3))]
    return rng, M, N, K, pad_a, pad_b, alpha, beta, out


@pytest.mark.parametrize("seed", range(24))
def test_random_16bit(orc, seed):
    import linear_layer_gb300 as ll
    rng, M, N, K, pad_a, pad_b, alpha, beta, out = _case(seed)
    kind = "f16" if seed % 2 == 0 else "bf16"
    lda, ldb = K + pad_a, N + pad_b
    A = wl.operand(kind, M, K, 100 + seed, ld=lda)
    B = wl.operand(kind, K, N, 200 + seed, ld=ldb)
    C = wl.f32_normal(M, N, 300 + seed) if beta != 0.0 else None
    tD = out_tensor(M, N, out)
    in_type = ll.IN_F16 if kind == "f16" else ll.IN_BF16
    noalloc = kind == "f16" and seed % 4 == 0
    if noalloc:
        ll.gemm_f16_noalloc(M, N, K, alpha, up(A), lda, up(B), ldb, beta, up(C), N, tD, N, out_code(out))
    else:
        need = ll.gemm_workspace_size(M, N, K, lda, ldb, in_type)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None
        fn = ll.gemm_f16 if kind == "f16" else ll.gemm_bf16
        fn(M, N, K, alpha, up(A), lda, up(B), ldb, beta, up(C), N, tD, N, out_code(out), workspace=ws)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, word
    what = "seed %d %s %dx%dx%d lda %d ldb %d a %g b %g %s%s" % (
        seed, kind, M, N, K, lda, ldb, alpha, beta, out, " noalloc" if noalloc else "")
    assert_fully_written(tD, M, N, what)
    Cf = None if C is None else C.ravel()
    check_all_rows(tD.float().cpu().numpy(),
                   lambda r: orc.gemm(kind, M, N, K, alpha, A.ravel(), lda, B.ravel(), ldb, beta, Cf, N, rows=r),
                   M, N, K, out, kind, what)


@pytest.mark.parametrize("seed", range(16))
def test_random_fp8(orc, seed):
    import linear_layer_gb300 as ll
    rng, M, N, K, pad_a, pad_b, alpha, beta, out = _case(100 + seed)
    a_fmt = ["e4m3", "e5m2"][seed % 2]
    b_fmt = ["e4m3", "e5m2"][(seed // 2) % 2]
    lda, ldb = K + pad_a, N + pad_b
    A, sA = wl.e4m3_blockquant_rowblocks(M, K, 400 + seed, ld=lda, fmt=a_fmt)
    B, sB = wl.e4m3_blockquant(K, N, 500 + seed, 128, 128, ld=ldb, fmt=b_fmt)
    C = wl.f32_normal(M, N, 600 + seed) if beta != 0.0 else None
    KB, NB = sA.shape[1], sB.shape[1]
    tD = out_tensor(M, N, out)
    need = ll.gemm_workspace_size(M, N, K, lda, ldb, ll.IN_E4M3)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None
    code = {"e4m3": ll.IN_E4M3, "e5m2": ll.IN_E5M2}
    ll.gemm_f8_blockscaled_mixed(code[a_fmt], code[b_fmt], M, N, K, alpha, up(A), lda, up(sA), KB, up(B), ldb,
                                 up(sB), NB, beta, up(C), N, tD, N, out_code(out), workspace=ws)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, word
    what = "seed %d %s x %s %dx%dx%d lda %d ldb %d a %g b %g %s" % (
        seed, a_fmt, b_fmt, M, N, K, lda, ldb, alpha, beta, out)
    assert_fully_written(tD, M, N, what)
    Cf = None if C is None else C.ravel()
    check_all_rows(tD.float().cpu().numpy(),
                   lambda r: orc.gemm_f8_blockscaled_mixed(a_fmt, b_fmt, M, N, K, alpha, A.ravel(), lda, sA.ravel(),
                                                           KB, B.ravel(), ldb, sB.ravel(), NB, beta, Cf, N, rows=r),
                   M, N, K, out, "e4m3", what)


@pytest.mark.parametrize("seed", range(16))
def test_random_pair_epilogues(orc, seed):
    """CTA-pair sizes with random C / D pitches (16-byte rows take the TMA epilogue, odd
    ones the transposing one), M and N tails inside a chunk, beta 0 or not, every output
    type, and in place (D == C) for some FP32 cases.  Rows past M and padding columns of
    D must stay untouched."""
    import linear_layer_gb300 as ll
    rng = np.random.default_rng(7000 + seed)
    M = int(rng.integers(1600, 4200))
    N = int(rng.integers(1600, 4200))
    K = int(rng.integers(16, 600))
    kind = "f16" if seed % 2 == 0 else "bf16"
    pad_a = int(rng.choice([0, 8, 3]))
    pad_b = int(rng.choice([0, 8, 5]))
    pad_cd = int(rng.choice([0, 0, 4, 8, 1, 3]))
    alpha = float(rng.choice([1.0, 0.5, -2.0]))
    beta = float(rng.choice([0.0, 1.0, -0.75]))
    out = OUTS[int(rng.integers(0, 3))]
    in_place = out == "f32" and beta != 0.0 and seed % 3 == 0
    lda, ldb, ldcd = K + pad_a, N + pad_b, N + pad_cd
    A = wl.operand(kind, M, K, 800 + seed, ld=lda)
    B = wl.operand(kind, K, N, 900 + seed, ld=ldb)
    C = wl.f32_normal(M, N, 1000 + seed, ld=ldcd) if beta != 0.0 else None
    guard = 8
    in_type = ll.IN_F16 if kind == "f16" else ll.IN_BF16
    need = ll.gemm_workspace_size(M, N, K, lda, ldb, in_type)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None
    fn = ll.gemm_f16 if kind == "f16" else ll.gemm_bf16
    if in_place:
        tC = torch.full((M + guard, ldcd), float("nan"), device="cuda")
        tC[:M] = up(C)
        fn(M, N, K, alpha, up(A), lda, up(B), ldb, beta, tC, ldcd, tC, ldcd, ll.OUT_F32, workspace=ws)
        tD = tC
    else:
        tD = out_tensor(M + guard, ldcd, out)
        fn(M, N, K, alpha, up(A), lda, up(B), ldb, beta, up(C), ldcd, tD, ldcd, out_code(out), workspace=ws)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, word
    D = tD.float().cpu().numpy()
    assert np.isnan(D[M:]).all(), "rows past M were written"
    if ldcd > N:  # (in place: C's padding is NaN too)
        assert np.isnan(D[:M, N:]).all(), "padding columns were written"
    what = "seed %d %s %dx%dx%d lda %d ldb %d ldcd %d a %g b %g %s%s" % (
        seed, kind, M, N, K, lda, ldb, ldcd, alpha, beta, out, " in place" if in_place else "")
    assert_fully_written(tD, M, N, what)
    Cf = None if C is None else C.ravel()
    check_all_rows(D, lambda r: orc.gemm(kind, M, N, K, alpha, A.ravel(), lda, B.ravel(), ldb, beta, Cf, ldcd,
                                         rows=r), M, N, K, out, kind, what)
