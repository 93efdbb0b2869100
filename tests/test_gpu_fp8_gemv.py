"""GPU parity of the FP8 block-scaled GEMM (tolerance bar; the full-size workload on every
element) and of the W8A8 GEMV (bit-exact z and y) against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import assert_fully_written, check_all_rows, check_close, out_code, out_tensor, up

pytestmark = pytest.mark.gpu


def run_fp8(orc, M, N, K, alpha=1.0, beta=0.0, out="bf16", pad=0, rows=None, seed=0):
    import linear_layer_gb300 as ll
    lda, ldb, ldc, ldd = K + pad, N + pad, N, N
    A, sA = wl.e4m3_blockquant_rowblocks(M, K, wl.SEED_A + seed, ld=lda)
    B, sB = wl.e4m3_blockquant(K, N, wl.SEED_B + seed, 128, 128, ld=ldb)
    C = wl.f32_normal(M, N, wl.SEED_C + seed) if beta != 0.0 else None
    KB, NB = sA.shape[1], sB.shape[1]
    tD = out_tensor(M, ldd, out)
    need = ll.gemm_workspace_size(M, N, K, lda, ldb, ll.IN_E4M3)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None
    ll.gemm_fp8_blockscaled(M, N, K, alpha, up(A), lda, up(sA), KB, up(B), ldb, up(sB), NB, beta,
                            up(C), ldc, tD, ldd, out_code(out), workspace=ws)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, "device status %s (word %#x)" % (ll.status_string(st), word)
    what = "fp8 %dx%dx%d" % (M, N, K)
    assert_fully_written(tD, M, N, what)
    D = tD.float().cpu().numpy()
    Cf = None if C is None else C.ravel()

    def oracle_rows(r):
        return orc.gemm_fp8_blockscaled(M, N, K, alpha, A.ravel(), lda, sA.ravel(), KB, B.ravel(), ldb,
                                        sB.ravel(), NB, beta, Cf, ldc, rows=r)
    if rows is None:  # every element, a chunk of rows at a time
        check_all_rows(D, oracle_rows, M, N, K, out, "e4m3", what)
    else:
        ref, absab = oracle_rows(rows)
        check_close(D[rows].astype(np.float64), ref, absab, K, out, "e4m3", what=what)


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (200, 300, 389), (1, 1, 1), (257, 513, 640),
                                   (64, 128, 1000)])
def test_fp8_small(orc, M, N, K):
    run_fp8(orc, M, N, K)


@pytest.mark.parametrize("out", ["f32", "f16"])
def test_fp8_alpha_beta_outputs(orc, out):
    run_fp8(orc, 260, 384, 300, alpha=0.5, beta=-1.25, out=out)


def test_fp8_padded_lds(orc):
    run_fp8(orc, 150, 270, 256, pad=16)


def test_fp8_unaligned_pitch_repacked(orc):
    run_fp8(orc, 100, 200, 200, pad=3)


@pytest.mark.parametrize("M,N,K,alpha,beta,out", [(2400, 2125, 1000, 1.0, 0.0, "bf16"),
                                                 (1200, 2200, 520, 1.0, 0.0, "bf16"),
                                                 (1300, 2049, 384, 0.5, -1.25, "f32"),
                                                 (2560, 2100, 256, 1.0, 0.0, "bf16")])
def test_fp8_wide_tiles(orc, M, N, K, alpha, beta, out):
    """Sizes that run 128 x 256 tiles: an odd number of 128-row blocks, more and fewer
    tiles than SMs, K tails, an N tail inside a 128-column block, and a last column block
    whose second half lies wholly past N."""
    run_fp8(orc, M, N, K, alpha, beta, out)


def test_fp8_8192_full_size(orc):
    """The FP8 workload at full size, every element (about 1.1e12 oracle multiply-adds)."""
    cfg = wl.WORKLOADS["e4m3_gemm_8192"]
    run_fp8(orc, cfg["M"], cfg["N"], cfg["K"], cfg["alpha"], cfg["beta"], cfg["out"])


# ------------------------------------------------------------------ W8A8 GEMV


def run_gemv(orc, N, K, ldw=None, x=None, W=None):
    import linear_layer_gb300 as ll
    ldw = K if ldw is None else ldw
    xg, sx, Wg, sW = wl.gemv_inputs(N, K, ldw)
    x = xg if x is None else x
    W = Wg if W is None else W
    ty = torch.full((N,), float("nan"), dtype=torch.float16, device="cuda")
    tz = torch.zeros(N, dtype=torch.int32, device="cuda")
    ll.linear_w8a8_gemv(N, K, up(x), torch.tensor([sx], device="cuda"), up(W), ldw, up(sW), ty, tz)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, "device status %s (word %#x)" % (ll.status_string(st), word)
    z_ref, y_ref = orc.gemv_w8a8(N, K, x, sx, W, ldw, sW)
    assert np.array_equal(tz.cpu().numpy().astype(np.int64), z_ref)
    assert np.array_equal(ty.cpu().numpy().view(np.uint16), y_ref.view(np.uint16))


def test_gemv_full_size_bit_exact(orc):
    cfg = wl.WORKLOADS["w8a8_gemv_4096x11008"]
    run_gemv(orc, cfg["N"], cfg["K"])


@pytest.mark.parametrize("N,K,ldw", [(1, 4096, 4096), (37, 4096, 4112), (300, 2048, 2048),
                                     (100, 16, 16), (64, 32768, 32768), (9, 100, 112), (33, 7, 7),
                                     (20, 0, 0), (5, 40000, 40000)])
def test_gemv_shapes(orc, N, K, ldw):
    run_gemv(orc, N, K, ldw)


def test_gemv_extreme_codes(orc):
    N, K = 3, 4096
    x = np.full(K, -128, np.int8)
    W = np.full((N, K), -128, np.int8)
    W[1] = 127
    W[2, ::2] = 127
    run_gemv(orc, N, K, x=x, W=W)


def test_gemv_without_z_out(orc):
    import linear_layer_gb300 as ll
    N, K = 50, 4096
    x, sx, W, sW = wl.gemv_inputs(N, K)
    ty = torch.empty(N, dtype=torch.float16, device="cuda")
    ll.linear_w8a8_gemv(N, K, up(x), torch.tensor([sx], device="cuda"), up(W), K, up(sW), ty, None)
    torch.cuda.synchronize()
    _, y_ref = orc.gemv_w8a8(N, K, x, sx, W, K, sW)
    assert np.array_equal(ty.cpu().numpy().view(np.uint16), y_ref.view(np.uint16))


def test_gemv_rejects_overflowing_k():
    import linear_layer_gb300 as ll
    t = torch.zeros(16, dtype=torch.int8, device="cuda")
    f = torch.zeros(16, dtype=torch.float32, device="cuda")
    with pytest.raises(ll.LLError) as e:
        ll.linear_w8a8_gemv(1, 131072, t, f, t, 131072, f, f, None)
    assert e.value.status == ll.LL_ERR_INVALID_ARG


@pytest.mark.parametrize("a_fmt,b_fmt", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
@pytest.mark.parametrize("M,N,K", [(200, 300, 389), (2048, 2048, 512), (2560, 2560, 1024)])
def test_f8_mixed_formats(orc, a_fmt, b_fmt, M, N, K):
    """Every pairing of E4M3 / E5M2 operands; 2560 x 2560 x 1024 (200 tiles of 128 x 256 on
    152 SMs) also splits its last wave by K ranges, the workspace query counting the slots."""
    import linear_layer_gb300 as ll
    code = {"e4m3": ll.IN_E4M3, "e5m2": ll.IN_E5M2}
    A, sA = wl.e4m3_blockquant_rowblocks(M, K, 61, fmt=a_fmt)
    B, sB = wl.e4m3_blockquant(K, N, 62, 128, 128, fmt=b_fmt)
    C = wl.f32_normal(M, N, 63)
    KB, NB = sA.shape[1], sB.shape[1]
    tD = out_tensor(M, N, "f32")
    need = ll.gemm_workspace_size(M, N, K, K, N, ll.IN_E4M3)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None
    ll.gemm_f8_blockscaled_mixed(code[a_fmt], code[b_fmt], M, N, K, 0.5, up(A), K, up(sA), KB, up(B),
                                 N, up(sB), NB, 1.5, up(C), N, tD, N, ll.OUT_F32, workspace=ws)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, word
    what = "%s x %s %dx%dx%d" % (a_fmt, b_fmt, M, N, K)
    assert_fully_written(tD, M, N, what)
    check_all_rows(tD.cpu().numpy(),
                   lambda r: orc.gemm_f8_blockscaled_mixed(a_fmt, b_fmt, M, N, K, 0.5, A.ravel(), K, sA.ravel(),
                                                           KB, B.ravel(), N, sB.ravel(), NB, 1.5, C.ravel(), N,
                                                           rows=r),
                   M, N, K, "f32", "e4m3", what)


def test_f8_mixed_rejects_16bit_types():
    import linear_layer_gb300 as ll
    t = torch.zeros(64, dtype=torch.uint8, device="cuda")
    f = torch.zeros(64, dtype=torch.float32, device="cuda")
    with pytest.raises(ll.LLError) as e:
        ll.gemm_f8_blockscaled_mixed(ll.IN_F16, ll.IN_E4M3, 4, 4, 4, 1.0, t, 4, f, 1, t, 4, f, 1, 0.0,
                                     None, 4, f, 4, ll.OUT_F32)
    assert e.value.status == ll.LL_ERR_INVALID_ARG
