"""GPU parity of the NVFP4 block-scaled GEMM (ll_gemm_nvf4: FP4 E2M1 elements, one UE4M3
scale per 16 K elements, applied by the tensor cores) against the CPU oracle, every element:
tails in M, N and K (K not a multiple of 16, 64 or 256), padded and TMA-illegal pitches
(repacked), scale matrices with padded pitches and rows that do not start on 4-byte
boundaries, alpha / beta and every output type, both kernels (one CTA per 128 x 256 tile for
small problems, CTA pairs per 256 x 256 tile for large ones), and the full-size 8192^3
workload.

Tolerance.  Every scaled element is an E2M1 value (2 significant bits) times a UE4M3 scale
(4 significant bits), so each product has at most 12 significant bits and lies between 2^-22
and 2^23: it is exact in FP32.  The only error is the FP32 accumulation over K, bounded by
about K u |a||b| (u = 2^-24) for any summation order; the test allows
NVF4_REL * sum_k |a_k b_k| per element (NVF4_REL = 2^-9, far above that bound at these
sizes, to leave room for an accumulator narrower than FP32 inside the tensor cores) plus the
output rounding, and a relative Frobenius error of at most NVF4_FROB."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import U_OUT, assert_fully_written, out_code, out_tensor, up

pytestmark = pytest.mark.gpu

NVF4_REL = 2.0 ** -9
NVF4_FROB = 1e-4
NAN_CODE = 0x7F   # UE4M3 NaN: pitch padding that would poison D if it were read


def check_nvf4_rows(D, oracle_rows, M, N, out, what, chunk=512):
    num = den = 0.0
    worst = 0.0
    for r0 in range(0, M, chunk):
        rows = np.arange(r0, min(M, r0 + chunk), dtype=np.int32)
        ref, absab = oracle_rows(rows)
        Dc = D[rows, :N].astype(np.float64)
        err = np.abs(Dc - ref)
        bound = NVF4_REL * absab + 1e-30 + U_OUT[out] * np.abs(ref)
        bad = ~(err <= bound)
        if bad.any():
            i, j = np.argwhere(bad)[0]
            raise AssertionError("%s: %d elements outside tolerance, e.g. (%d, %d): got %r want %r bound %r"
                                 % (what, int(bad.sum()), r0 + i, j, Dc[i, j], ref[i, j], bound[i, j]))
        if out == "f32":
            worst = max(worst, float(np.max(err / np.maximum(absab, 1e-30))))
        num += float(np.sum((Dc - ref) ** 2))
        den += float(np.sum(ref ** 2))
    if den > 0:
        rel = np.sqrt(num / den)
        bar = NVF4_FROB + U_OUT[out] * (1.0 + NVF4_FROB)
        assert rel <= bar, "%s: relative Frobenius error %g > %g" % (what, rel, bar)
    if out == "f32":
        print("%s: max |err| / sum|ab| = %.3g" % (what, worst))


def run_nvf4(orc, M, N, K, alpha=1.0, beta=0.0, out="bf16", pad=0, spad=0, soff=0, seed=0):
    import linear_layer_gb300 as ll
    lda = ldbt = K + pad                       # pitches in elements (even)
    A, SA = wl.nvf4_quant(M, K, 1700 + seed, ld=lda)
    Bt, SB = wl.nvf4_quant(N, K, 1800 + seed, ld=ldbt)
    KB = SA.shape[1]
    ld_s = KB + spad
    SAp = np.full((M, ld_s), NAN_CODE, np.uint8)
    SAp[:, :KB] = SA
    SBp = np.full((N, ld_s), NAN_CODE, np.uint8)
    SBp[:, :KB] = SB
    C = wl.f32_normal(M, N, 1900 + seed) if beta != 0.0 else None
    tD = out_tensor(M, N, out)
    tSA = torch.empty(SAp.size + 16, dtype=torch.uint8, device="cuda")
    tSA[soff:soff + SAp.size] = up(SAp.ravel())
    tSB = torch.empty(SBp.size + 16, dtype=torch.uint8, device="cuda")
    tSB[soff:soff + SBp.size] = up(SBp.ravel())
    need = ll.gemm_nvf4_workspace_size(M, N, K, lda, ldbt)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ll.gemm_nvf4(M, N, K, alpha, up(A), lda, tSA.data_ptr() + soff, ld_s, up(Bt), ldbt, tSB.data_ptr() + soff,
                 ld_s, beta, up(C), N, tD, N, out_code(out), workspace=ws)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, "device status %s (word %#x)" % (ll.status_string(st), word)
    what = "nvf4 %dx%dx%d %s" % (M, N, K, out)
    assert_fully_written(tD, M, N, what)
    Cf = None if C is None else C.ravel()
    check_nvf4_rows(tD.float().cpu().numpy(),
                    lambda r: orc.gemm_nvf4(M, N, K, alpha, A.ravel(), lda, SAp.ravel(), ld_s, Bt.ravel(), ldbt,
                                            SBp.ravel(), ld_s, beta, Cf, N, rows=r),
                    M, N, out, what)
    return tD


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (128, 256, 64), (200, 300, 390), (1, 1, 2), (257, 513, 640),
                                   (64, 128, 1000), (300, 700, 78), (1024, 1024, 1024), (130, 260, 16)])
def test_nvf4_shapes(orc, M, N, K):
    run_nvf4(orc, M, N, K, out="f32")


@pytest.mark.parametrize("out", ["f32", "f16", "bf16"])
def test_nvf4_alpha_beta_outputs(orc, out):
    run_nvf4(orc, 260, 384, 300, alpha=0.5, beta=-1.25, out=out)


def test_nvf4_padded_and_repacked_pitches(orc):
    run_nvf4(orc, 150, 270, 512, pad=32, spad=3, out="f32")   # padded 16-byte pitches (272 bytes)
    run_nvf4(orc, 100, 200, 200, pad=2, spad=1, out="f32")    # 101-byte rows: A and Bt repacked


def test_nvf4_unaligned_scale_rows(orc):
    run_nvf4(orc, 130, 260, 768, spad=1, soff=1, out="f32")
    run_nvf4(orc, 130, 260, 768, spad=0, soff=3, out="f32")
    run_nvf4(orc, 130, 260, 4096, spad=0, out="f32")          # 256 codes a row: read in place


def test_nvf4_many_tiles(orc):
    run_nvf4(orc, 2000, 1000, 512, beta=1.0, out="f32", seed=5)


@pytest.mark.parametrize("M,N,K,alpha,beta,out,spad", [
    (2100, 2600, 778, 0.5, -1.25, "f32", 0),
    (4096, 2048, 1024, 1.0, 0.0, "bf16", 0),
    (1999, 4100, 256, 1.0, 1.0, "f16", 3),
    (2304, 2304, 4096, 1.0, 0.0, "f32", 0)])
def test_nvf4_pair_kernel(orc, M, N, K, alpha, beta, out, spad):
    """Sizes with at least a quarter of the SM pairs' worth of 256 x 256 tiles run on CTA
    pairs: M tails inside the odd CTA's rows, N tails inside a row half of Bt, K tails,
    alpha / beta, every output type, repacked scale matrices."""
    run_nvf4(orc, M, N, K, alpha, beta, out, spad=spad, seed=11)


def test_nvf4_needs_workspace():
    import linear_layer_gb300 as ll
    M = N = K = 256
    t = torch.zeros(M * K // 2, dtype=torch.uint8, device="cuda")
    s = torch.full((M * 16,), 0x38, dtype=torch.uint8, device="cuda")
    D = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    need = ll.gemm_nvf4_workspace_size(M, N, K, K, K)
    for ws in (None, torch.empty(need - 1, dtype=torch.uint8, device="cuda")):
        with pytest.raises(ll.LLError) as e:
            ll.gemm_nvf4(M, N, K, 1.0, t, K, s, 16, t, K, s, 16, 0.0, None, N, D, N, ll.OUT_BF16, workspace=ws)
        assert e.value.status == ll.LL_ERR_WORKSPACE


def test_nvf4_deterministic(orc):
    a = run_nvf4(orc, 512, 768, 512, seed=7)
    b = run_nvf4(orc, 512, 768, 512, seed=7)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_nvf4_8192_full_size(orc):
    """The NVFP4 workload at full size (8192^3, BF16 out), every element."""
    cfg = wl.WORKLOADS["nvf4_gemm_8192"]
    run_nvf4(orc, cfg["M"], cfg["N"], cfg["K"], cfg["alpha"], cfg["beta"], cfg["out"])


def test_nvf4_k_zero_is_beta_c():
    """K = 0: an empty contraction, D = beta * C exactly (no scale codes or workspace read)."""
    import linear_layer_gb300 as ll
    M, N = 300, 260
    C = wl.f32_normal(M, N, 77)
    tD = out_tensor(M, N, "f32")
    ll.gemm_nvf4(M, N, 0, 1.0, None, 0, None, 0, None, 0, None, 0, -0.75, up(C), N, tD, N, ll.OUT_F32)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK
    want = torch.from_numpy((np.float32(-0.75) * C).astype(np.float32))
    assert torch.equal(tD.cpu(), want)


@pytest.mark.parametrize("M,N,K,alpha,beta,out", [(2560, 2500, 2300, 1.0, 1.0, "f16"),
                                                  (2500, 2560, 2048, 0.5, 0.0, "f32")])
def test_nvf4_pair_kernel_partial_wave(orc, M, N, K, alpha, beta, out):
    """100 pair tiles on the CTA-pair kernel: more than a wave of SM pairs, then a partial
    one, with M, N and K tails (8 or 9 K blocks of 256)."""
    run_nvf4(orc, M, N, K, alpha, beta, out, seed=13)
