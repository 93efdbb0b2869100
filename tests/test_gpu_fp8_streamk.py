"""GPU parity of the one-CTA FP8 block-scaled GEMM when its last partial wave of 128 x 256
tiles is split by K ranges across all CTAs (stream-K; used when the caller's workspace has
room for the promoted partial tiles, ll_gemm_workspace_size counting them): every element
against the oracle for tails in M, N and K, alpha / beta and the output types; outputs
bit-identical from run to run; and one byte less workspace turning the split off (then
bit-identical to the call without workspace).  The full-size 8192^3 case in
test_gpu_fp8_gemv.py runs the split as well (13 whole waves and 72 more tiles)."""
import pytest
import torch

import workloads as wl
from gpu_util import assert_fully_written, check_all_rows, out_code, out_tensor, up

pytestmark = pytest.mark.gpu


def _inputs(M, N, K, beta, seed):
    A, sA = wl.e4m3_blockquant_rowblocks(M, K, wl.SEED_A + seed)
    B, sB = wl.e4m3_blockquant(K, N, wl.SEED_B + seed, 128, 128)
    C = wl.f32_normal(M, N, wl.SEED_C + seed) if beta != 0.0 else None
    return A, sA, B, sB, C


def _call(M, N, K, alpha, beta, out, inp, ws):
    import linear_layer_gb300 as ll
    A, sA, B, sB, C = inp
    tD = out_tensor(M, N, out)
    ll.gemm_fp8_blockscaled(M, N, K, alpha, up(A), K, up(sA), sA.shape[1], up(B), N, up(sB), sB.shape[1], beta,
                            up(C), N, tD, N, out_code(out), workspace=ws)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, "device status %s (word %#x)" % (ll.status_string(st), word)
    return tD


# 200 tiles of 128 x 256 on 152 CTAs: one whole wave and 48 tiles split by K (8 or 9 K
# blocks a tile, about three pieces each)
@pytest.mark.parametrize("M,N,K,alpha,beta,out", [
    (2560, 2560, 1024, 1.0, 0.0, "bf16"),
    (2500, 2400, 1100, 0.5, -1.25, "f32"),
    (2560, 2500, 1408, 1.0, 1.0, "f16")])
def test_fp8_streamk_tail(orc, M, N, K, alpha, beta, out):
    import linear_layer_gb300 as ll
    need = ll.gemm_workspace_size(M, N, K, K, N, ll.IN_E4M3)
    assert need > 0  # the workspace size counts the partial tiles
    inp = _inputs(M, N, K, beta, 7)
    tD = _call(M, N, K, alpha, beta, out, inp, torch.empty(need, dtype=torch.uint8, device="cuda"))
    what = "fp8 stream-K %dx%dx%d" % (M, N, K)
    assert_fully_written(tD, M, N, what)
    A, sA, B, sB, C = inp
    Cf = None if C is None else C.ravel()
    check_all_rows(tD.float().cpu().numpy(),
                   lambda r: orc.gemm_fp8_blockscaled(M, N, K, alpha, A.ravel(), K, sA.ravel(), sA.shape[1],
                                                      B.ravel(), N, sB.ravel(), sB.shape[1], beta, Cf, N, rows=r),
                   M, N, K, out, "e4m3", what)


def test_fp8_streamk_deterministic_and_opt_out():
    import linear_layer_gb300 as ll
    M, N, K = 2560, 2560, 1024
    inp = _inputs(M, N, K, 1.0, 9)
    need = ll.gemm_workspace_size(M, N, K, K, N, ll.IN_E4M3)
    full = torch.empty(need, dtype=torch.uint8, device="cuda")
    a = _call(M, N, K, 1.0, 1.0, "f32", inp, full)
    b = _call(M, N, K, 1.0, 1.0, "f32", inp, full)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    c = _call(M, N, K, 1.0, 1.0, "f32", inp, None)
    d = _call(M, N, K, 1.0, 1.0, "f32", inp, torch.empty(need - 1, dtype=torch.uint8, device="cuda"))
    assert torch.equal(c.view(torch.int32), d.view(torch.int32))
