"""GPU parity of the MX block-scaled 8-bit GEMM (ll_gemm_mxf8, hardware block scaling on the
tensor cores) against the CPU oracle, every element, at the FP8 tolerance bar: tails in M, N
and K (K not a multiple of 32 or 128), padded operand and scale pitches, TMA-illegal pitches
(repacked), scale matrices whose rows do not start on 4-byte boundaries, alpha / beta and
every output type, E4M3 and E5M2 elements, both kernels (one CTA per 128 x 256 tile for
small problems, CTA pairs per 256 x 256 tile for large ones), and the full-size 8192^3
workload."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import assert_fully_written, check_all_rows, out_code, out_tensor, up

pytestmark = pytest.mark.gpu


def run_mx(orc, M, N, K, alpha=1.0, beta=0.0, out="bf16", pad=0, spad=0, soff=0, a_fmt="e4m3", b_fmt="e4m3",
           seed=0):
    import linear_layer_gb300 as ll
    lda, ldb = K + pad, N + pad
    A, SA = wl.mx_quant(M, K, 700 + seed, 1, ld=lda, fmt=a_fmt)
    B, SB = wl.mx_quant(K, N, 800 + seed, 0, ld=ldb, fmt=b_fmt)
    KB = SA.shape[1]
    ld_s = KB + spad
    SAp = np.full((M, ld_s), 250, np.uint8)   # padding codes that would be visibly wrong if read
    SAp[:, :KB] = SA
    SBp = np.full((N, ld_s), 250, np.uint8)
    SBp[:, :KB] = SB
    C = wl.f32_normal(M, N, 900 + seed) if beta != 0.0 else None
    tD = out_tensor(M, N, out)
    # scale matrices `soff` bytes past an aligned start
    tSA = torch.empty(SAp.size + 16, dtype=torch.uint8, device="cuda")
    tSA[soff:soff + SAp.size] = up(SAp.ravel())
    tSB = torch.empty(SBp.size + 16, dtype=torch.uint8, device="cuda")
    tSB[soff:soff + SBp.size] = up(SBp.ravel())
    need = ll.gemm_mxf8_workspace_size(M, N, K, lda, ldb)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda") if need else None
    code = {"e4m3": ll.IN_E4M3, "e5m2": ll.IN_E5M2}
    ll.gemm_mxf8(code[a_fmt], code[b_fmt], M, N, K, alpha, up(A), lda, tSA.data_ptr() + soff, ld_s, up(B), ldb,
                 tSB.data_ptr() + soff, ld_s, beta, up(C), N, tD, N, out_code(out), workspace=ws)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, "device status %s (word %#x)" % (ll.status_string(st), word)
    what = "mx %s x %s %dx%dx%d" % (a_fmt, b_fmt, M, N, K)
    assert_fully_written(tD, M, N, what)
    Cf = None if C is None else C.ravel()
    check_all_rows(tD.float().cpu().numpy(),
                   lambda r: orc.gemm_mx_f8(a_fmt, b_fmt, M, N, K, alpha, A.ravel(), lda, SAp.ravel(), ld_s,
                                            B.ravel(), ldb, SBp.ravel(), ld_s, beta, Cf, N, rows=r),
                   M, N, K, out, "e4m3", what)
    return tD


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (128, 256, 32), (200, 300, 389), (1, 1, 1), (257, 513, 640),
                                   (64, 128, 1000), (300, 700, 77), (1024, 1024, 1024)])
def test_mx_shapes(orc, M, N, K):
    run_mx(orc, M, N, K)


@pytest.mark.parametrize("out", ["f32", "f16", "bf16"])
def test_mx_alpha_beta_outputs(orc, out):
    run_mx(orc, 260, 384, 300, alpha=0.5, beta=-1.25, out=out)


@pytest.mark.parametrize("a_fmt,b_fmt", [("e5m2", "e5m2"), ("e4m3", "e5m2"), ("e5m2", "e4m3")])
def test_mx_element_formats(orc, a_fmt, b_fmt):
    run_mx(orc, 300, 520, 416, a_fmt=a_fmt, b_fmt=b_fmt, seed=3)


def test_mx_padded_and_repacked_pitches(orc):
    run_mx(orc, 150, 270, 256, pad=16, spad=3)   # padded, 16-byte pitches
    run_mx(orc, 100, 200, 200, pad=3, spad=1)    # TMA-illegal pitches: A and B repacked


def test_mx_unaligned_scale_rows(orc):
    # scale matrices 1 and 3 bytes past an aligned start, pitches that are not a multiple of
    # 16 bytes, and 16-byte pitches (read with 16-byte loads when rearranged)
    run_mx(orc, 130, 260, 384, spad=1, soff=1)
    run_mx(orc, 130, 260, 384, spad=0, soff=3)
    run_mx(orc, 130, 260, 384, spad=5)
    run_mx(orc, 130, 260, 2048, spad=0)      # 64 K blocks: a 64-byte pitch, in place


def test_mx_many_tiles(orc):
    # more tiles than SMs (several per CTA) with M and N tails
    run_mx(orc, 2000, 3000, 512, beta=1.0, out="f32", seed=5)


@pytest.mark.parametrize("M,N,K,alpha,beta,out,a_fmt,b_fmt,spad", [
    (2100, 2600, 777, 0.5, -1.25, "f32", "e4m3", "e4m3", 0),
    (4096, 2048, 1024, 1.0, 0.0, "bf16", "e5m2", "e4m3", 0),
    (1999, 4100, 256, 1.0, 1.0, "f16", "e4m3", "e5m2", 3),
    (2304, 2304, 4096, 1.0, 0.0, "bf16", "e4m3", "e4m3", 0)])
def test_mx_pair_kernel(orc, M, N, K, alpha, beta, out, a_fmt, b_fmt, spad):
    """Sizes with at least a quarter of the SM pairs' worth of 256 x 256 tiles run on CTA
    pairs: M tails inside the odd CTA's rows, N tails inside a column half, K tails, mixed
    element formats, alpha / beta, every output type, repacked scale matrices."""
    run_mx(orc, M, N, K, alpha, beta, out, spad=spad, a_fmt=a_fmt, b_fmt=b_fmt, seed=11)


def test_mx_needs_workspace():
    """The rearranged scale codes always need workspace: a call without it, or with too
    little, is rejected before anything runs."""
    import linear_layer_gb300 as ll
    M = N = K = 256
    t = torch.zeros(M * K, dtype=torch.uint8, device="cuda")
    s = torch.full((M * 8,), 127, dtype=torch.uint8, device="cuda")
    D = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    need = ll.gemm_mxf8_workspace_size(M, N, K, K, N)
    for ws in (None, torch.empty(need - 1, dtype=torch.uint8, device="cuda")):
        with pytest.raises(ll.LLError) as e:
            ll.gemm_mxf8(ll.IN_E4M3, ll.IN_E4M3, M, N, K, 1.0, t, K, s, 8, t, N, s, 8, 0.0, None, N, D, N,
                         ll.OUT_BF16, workspace=ws)
        assert e.value.status == ll.LL_ERR_WORKSPACE


def test_mx_deterministic(orc):
    a = run_mx(orc, 512, 768, 512, seed=7)
    b = run_mx(orc, 512, 768, 512, seed=7)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_mx_8192_full_size(orc):
    """The MX FP8 workload at full size (8192^3, E4M3, BF16 out), every element."""
    cfg = wl.WORKLOADS["mxf8_gemm_8192"]
    run_mx(orc, cfg["M"], cfg["N"], cfg["K"], cfg["alpha"], cfg["beta"], cfg["out"])


def test_mx_k_zero_is_beta_c():
    """K = 0: an empty contraction, D = beta * C exactly (no scale codes or workspace read)."""
    import linear_layer_gb300 as ll
    M, N = 300, 260
    C = wl.f32_normal(M, N, 78)
    tD = out_tensor(M, N, "f32")
    ll.gemm_mxf8(ll.IN_E4M3, ll.IN_E4M3, M, N, 0, 1.0, None, 0, None, 0, None, N, None, 0, 2.5, up(C), N, tD, N,
                 ll.OUT_F32)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK
    want = torch.from_numpy((np.float32(2.5) * C).astype(np.float32))
    assert torch.equal(tD.cpu(), want)


@pytest.mark.parametrize("M,N,K,alpha,beta,out", [(2560, 2560, 1100, 0.5, -1.25, "f32"),
                                                  (2500, 2400, 1024, 1.0, 0.0, "bf16")])
def test_mx_pair_kernel_partial_wave(orc, M, N, K, alpha, beta, out):
    """100 pair tiles on the CTA-pair kernel: more than a wave of SM pairs, then a partial
    one, with K, M and N tails; repeat calls bit-identical."""
    a = run_mx(orc, M, N, K, alpha, beta, out, seed=13)
    b = run_mx(orc, M, N, K, alpha, beta, out, seed=13)
    assert torch.equal(a.view(torch.int32 if out == "f32" else torch.int16),
                       b.view(torch.int32 if out == "f32" else torch.int16))
