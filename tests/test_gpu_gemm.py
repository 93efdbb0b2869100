"""GPU parity of the FP16 / BF16 tcgen05 GEMM against the CPU oracle, through the C ABI.

Every test compares every element, the full-size workloads included (BF16 4096^3,
and the ragged FP16 4093 x 5003 x 2056 with tight and with padded leading
dimensions, in the launch configuration the benchmark times).  D is pre-filled with
NaN and every test checks that all of D[:M, :N] was written.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import assert_fully_written, check_all_rows, check_close, out_code, out_tensor, up

pytestmark = pytest.mark.gpu


def _dec_out(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_gemm(orc, kind, M, N, K, alpha, beta, out, lda=None, ldb=None, ldc=None, ldd=None,
             rows=None, seed_shift=0, A=None, B=None, C=None, workspace=True):
    import linear_layer_gb300 as ll
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    ldd = N if ldd is None else ldd
    if A is None:
        A = wl.operand(kind, M, K, wl.SEED_A + seed_shift, ld=lda)
        B = wl.operand(kind, K, N, wl.SEED_B + seed_shift, ld=ldb)
        C = wl.f32_normal(M, N, wl.SEED_C + seed_shift, ld=ldc) if beta != 0.0 else None
    tA, tB, tC = up(A), up(B), up(C)
    tD = out_tensor(M, ldd, out)
    in_type = ll.IN_F16 if kind == "f16" else ll.IN_BF16
    ws = None
    need = ll.gemm_workspace_size(M, N, K, lda, ldb, in_type)
    if need and workspace:
        ws = torch.empty(need, dtype=torch.uint8, device=tA.device)
    fn = ll.gemm_f16 if kind == "f16" else ll.gemm_bf16
    fn(M, N, K, alpha, tA, lda, tB, ldb, beta, tC, ldc, tD, ldd, out_code(out), workspace=ws)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, "device status %s (word %#x)" % (ll.status_string(st), word)
    what = "%s %dx%dx%d" % (kind, M, N, K)
    assert_fully_written(tD, M, N, what)
    D = _dec_out(tD)
    Cf = None if C is None else C.ravel()
    if rows is None:  # every element, a chunk of rows at a time
        check_all_rows(D, lambda r: orc.gemm(kind, M, N, K, alpha, A.ravel(), lda, B.ravel(), ldb, beta, Cf,
                                             ldc, rows=r), M, N, K, out, kind, what)
    else:
        ref, absab = orc.gemm(kind, M, N, K, alpha, A.ravel(), lda, B.ravel(), ldb, beta, Cf, ldc, rows=rows)
        check_close(D[rows, :N], ref, absab, K, out, kind, what=what)
    if ldd > N:  # padding columns of D are never written
        assert torch.isnan(tD[:, N:].float()).all()
    return D


def test_f16_256_cube_f32_out(orc):
    """The FP16 256^3 workload: C not read (beta = 0), FP32 output."""
    cfg = wl.WORKLOADS["f16_gemm_256"]
    run_gemm(orc, "f16", cfg["M"], cfg["N"], cfg["K"], cfg["alpha"], cfg["beta"], cfg["out"])


@pytest.mark.parametrize("kind", ["f16", "bf16"])
@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
def test_small_tails_all_outputs(orc, kind, out):
    # several tiles in M and N, ragged M / N / K tails, beta != 0
    run_gemm(orc, kind, 300, 520, 200, 0.75, -0.5, out)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 1, 16), (5, 7, 3), (129, 65, 64), (128, 256, 65),
                                   (64, 1000, 8), (700, 300, 1)])
def test_odd_shapes(orc, M, N, K):
    run_gemm(orc, "bf16", M, N, K, 1.0, 1.0, "f32")


def test_many_tiles_every_path(orc):
    # one-CTA 128 x 64 tiles, CTA-pair halves only (at most half a wave of pair tiles),
    # whole pair tiles, and an M of 128 (one-CTA kernel although it has 24 pair tiles)
    for (M, N) in [(256, 256), (1280, 1280), (2048, 1280), (4096, 2304), (128, 6144)]:
        run_gemm(orc, "f16", M, N, 128, 1.0, 0.0, "f32")


def test_padded_leading_dims(orc):
    run_gemm(orc, "f16", 200, 300, 136, 1.5, 0.25, "f32", lda=152, ldb=328, ldc=301, ldd=310)


def test_unaligned_pitch_needs_workspace(orc):
    import linear_layer_gb300 as ll
    with pytest.raises(ll.LLError) as e:
        run_gemm(orc, "f16", 64, 77, 40, 1.0, 0.0, "f32", ldb=77, workspace=False)
    assert e.value.status == ll.LL_ERR_WORKSPACE
    run_gemm(orc, "f16", 64, 77, 40, 1.0, 0.0, "f32", lda=41, ldb=77)


def test_k_zero_is_beta_c(orc):
    run_gemm(orc, "bf16", 70, 90, 0, 2.0, -1.25, "f32")
    run_gemm(orc, "bf16", 70, 90, 0, 2.0, 0.0, "bf16")


def test_in_place_c_equals_d(orc):
    import linear_layer_gb300 as ll
    M, N, K = 130, 144, 72  # 16-byte row pitches: read in place, no workspace
    A = wl.operand("f16", M, K, 7)
    B = wl.operand("f16", K, N, 8)
    C = wl.f32_normal(M, N, 9)
    tC = up(C)
    ll.gemm_f16(M, N, K, 1.0, up(A), K, up(B), N, 2.0, tC, N, tC, N, ll.OUT_F32)
    ref, absab = orc.gemm("f16", M, N, K, 1.0, A.ravel(), K, B.ravel(), N, 2.0, C.ravel(), N)
    check_close(tC.cpu().numpy(), ref, absab, K, "f32", "f16", "in place")


def test_deterministic(orc):
    import linear_layer_gb300 as ll
    M, N, K = 512, 768, 512
    A, B, C = wl.gemm_inputs("bf16", M, N, K, 1.0)
    tA, tB, tC = up(A), up(B), up(C)
    outs = []
    for _ in range(3):
        tD = out_tensor(M, N, "bf16")
        ll.gemm_bf16(M, N, K, 1.0, tA, K, tB, N, 1.0, tC, N, tD, N, ll.OUT_BF16)
        outs.append(tD.view(torch.int16).cpu().numpy())
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_invalid_args_rejected_before_launch():
    import linear_layer_gb300 as ll
    t = torch.zeros(64, dtype=torch.float16, device="cuda")
    D = torch.zeros(64, dtype=torch.float32, device="cuda")
    cases = [
        dict(M=-1, N=4, K=4, lda=4, ldb=4, C=None, beta=0.0, ldd=4),
        dict(M=4, N=4, K=4, lda=3, ldb=4, C=None, beta=0.0, ldd=4),
        dict(M=4, N=4, K=4, lda=4, ldb=4, C=None, beta=1.0, ldd=4),
        dict(M=4, N=4, K=4, lda=4, ldb=4, C=None, beta=0.0, ldd=3),
    ]
    for c in cases:
        with pytest.raises(ll.LLError) as e:
            ll.gemm_f16(c["M"], c["N"], c["K"], 1.0, t, c["lda"], t, c["ldb"], c["beta"], c["C"], 4,
                        D, c["ldd"], ll.OUT_F32)
        assert e.value.status == ll.LL_ERR_INVALID_ARG
    # M == 0 / N == 0 are no-ops
    ll.gemm_f16(0, 4, 4, 1.0, t, 4, t, 4, 0.0, None, 4, D, 4, ll.OUT_F32)
    ll.gemm_f16(4, 0, 4, 1.0, t, 4, t, 4, 0.0, None, 4, D, 4, ll.OUT_F32)


def test_bf16_4096_full_size(orc):
    """The headline workload at full size, every element."""
    cfg = wl.WORKLOADS["bf16_gemm_4096"]
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    run_gemm(orc, "bf16", M, N, K, cfg["alpha"], cfg["beta"], cfg["out"])


def test_bf16_4096_fp32_output_strict_bar(orc):
    # the same workload and kernel with an FP32 epilogue: the 1e-3 Frobenius bar
    # applies to the accumulator before any cast, with no allowance for it
    cfg = wl.WORKLOADS["bf16_gemm_4096"]
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    run_gemm(orc, "bf16", M, N, K, cfg["alpha"], cfg["beta"], "f32")


def test_f16_ragged_tight_lds_full_size(orc):
    """The ragged workload with tight leading dimensions (B repacked), every element."""
    cfg = wl.WORKLOADS["f16_gemm_4093x5003x2056"]
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    run_gemm(orc, "f16", M, N, K, cfg["alpha"], cfg["beta"], cfg["out"])


def test_f16_ragged_padded_lds_full_size(orc):
    cfg = wl.WORKLOADS["f16_gemm_4093x5003x2056"]
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    run_gemm(orc, "f16", M, N, K, cfg["alpha"], cfg["beta"], cfg["out"], lda=2064, ldb=5008,
             ldc=5008, ldd=5008)


def _shifted(t, shift, fill=0.0):
    """A flat device copy of t that starts `shift` elements into its buffer, so its base
    address is shift * element size bytes past an aligned boundary."""
    flat = t.reshape(-1)
    buf = torch.full((flat.numel() + shift,), fill, dtype=flat.dtype, device=flat.device)
    buf[shift:] = flat
    return buf[shift:]


@pytest.mark.parametrize("M,N,K", [(200, 136, 72), (1600, 1664, 136)])
def test_misaligned_base_pointers(orc, M, N, K):
    """A and B start 2 and 6 bytes past a 16-byte boundary (both are repacked); C and D
    start 4 bytes past one (the transposing epilogue with scalar accesses).  The second
    shape runs on CTA pairs."""
    import linear_layer_gb300 as ll
    A = wl.operand("f16", M, K, 41)
    B = wl.operand("f16", K, N, 42)
    C = wl.f32_normal(M, N, 43)
    tA, tB, tC = _shifted(up(A), 1), _shifted(up(B), 3), _shifted(up(C), 1)
    tD = _shifted(torch.empty(M * N, device="cuda"), 1, float("nan"))
    need = ll.gemm_workspace_size(M, N, K, 1, 1, ll.IN_F16)  # the misaligned-base bound
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ll.gemm_f16(M, N, K, 0.5, tA, K, tB, N, 1.5, tC, N, tD, N, ll.OUT_F32, workspace=ws)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, "device status %s (word %#x)" % (ll.status_string(st), word)
    ref, absab = orc.gemm("f16", M, N, K, 0.5, A.ravel(), K, B.ravel(), N, 1.5, C.ravel(), N)
    check_close(tD.reshape(M, N).cpu().numpy(), ref, absab, K, "f32", "f16", "misaligned bases")


@pytest.mark.parametrize("ld_pad", [0, 1])
@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
def test_pair_several_units_per_cta(orc, ld_pad, out):
    """CTA-pair problem with two whole waves plus half tiles, so each epilogue warp loads
    the next unit's first chunk of C ahead; 16-byte row pitches of C and D (rows stored
    per lane) and odd pitches (transposed through shared memory)."""
    M, N, K = 4096, 2560, 64
    ld = N + ld_pad
    run_gemm(orc, "bf16", M, N, K, 0.75, -1.5, out, ldc=ld, ldd=ld)


@pytest.mark.parametrize("ld_pad", [0, 1])
def test_pair_in_place_c_equals_d(orc, ld_pad):
    """D = alpha * A B + beta * D on CTA pairs, in both epilogue layouts."""
    import linear_layer_gb300 as ll
    M, N, K = 2048, 2304, 96
    ld = N + ld_pad
    A = wl.operand("bf16", M, K, 51)
    B = wl.operand("bf16", K, N, 52)
    C = wl.f32_normal(M, N, 53, ld=ld)
    tC = up(C)
    ll.gemm_bf16(M, N, K, 1.0, up(A), K, up(B), N, -0.5, tC, ld, tC, ld, ll.OUT_F32)
    assert_fully_written(tC, M, N, "pair in place")
    check_all_rows(tC.cpu().numpy(), lambda r: orc.gemm("bf16", M, N, K, 1.0, A.ravel(), K, B.ravel(), N, -0.5,
                                                        C.ravel(), ld, rows=r), M, N, K, "f32", "bf16", "pair in place")


@pytest.mark.parametrize("ldc,c_off", [(2001, 0), (2009, 8), (2003, 0), (2001, 1)])
def test_pair_fp32_rows_off_grid_c_pitches_and_offsets(orc, ldc, c_off):
    """FP32 D with 2001-float rows (off the 16- and 32-byte grids) on CTA pairs, C read
    through TMA by row classes with its own pitch and base offset (the same sector grid
    as D's rows, or another), D stored by whole sectors.  Every element, padding columns
    and rows past M untouched."""
    import linear_layer_gb300 as ll
    M, N, K, ldd = 1500, 1992, 200, 2001
    A = wl.operand("bf16", M, K, 71)
    B = wl.operand("bf16", K, N, 72)
    C = wl.f32_normal(M, N, 73, ld=ldc)
    buf = torch.full((M * ldc + 8,), float("nan"), dtype=torch.float32, device="cuda")
    buf[c_off:c_off + M * ldc] = up(C.ravel())
    tC = buf[c_off:c_off + M * ldc]
    guard = 9
    tD = out_tensor(M + guard, ldd, "f32")
    ll.gemm_bf16(M, N, K, 0.75, up(A), K, up(B), N, -1.25, tC, ldc, tD, ldd, ll.OUT_F32)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, "device status %s (word %#x)" % (ll.status_string(st), word)
    D = tD.cpu().numpy()
    assert np.isnan(D[M:]).all(), "rows past M were written"
    assert np.isnan(D[:M, N:]).all(), "padding columns were written"
    assert_fully_written(tD, M, N, "C pitch %d offset %d" % (ldc, c_off))
    check_all_rows(D, lambda r: orc.gemm("bf16", M, N, K, 0.75, A.ravel(), K, B.ravel(), N, -1.25, C.ravel(), ldc,
                                         rows=r), M, N, K, "f32", "bf16", "C pitch %d offset %d" % (ldc, c_off))


@pytest.mark.parametrize("ld_pad", [0, 8, 3])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_pair_writes_nothing_outside_d(orc, ld_pad, out):
    """M and N tails that end inside a 32-row / 32-column chunk, on CTA pairs: the rows
    after D's last row and the padding columns of every row stay untouched, with the
    TMA epilogue (16-byte row pitches: ld_pad 0 and 8) and the transposing one (odd
    pitch)."""
    import linear_layer_gb300 as ll
    M, N, K = 2000, 2264, 80
    ldd = N + ld_pad if out == "f32" else N + 2 * ld_pad
    A = wl.operand("bf16", M, K, 61)
    B = wl.operand("bf16", K, N, 62)
    C = wl.f32_normal(M, N, 63, ld=ldd)
    guard = 40  # rows past M in the same allocation
    tD = out_tensor(M + guard, ldd, out)
    ll.gemm_bf16(M, N, K, 1.0, up(A), K, up(B), N, 0.5, up(C), ldd, tD, ldd, out_code(out))
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, "device status %s (word %#x)" % (ll.status_string(st), word)
    D = tD.float().cpu().numpy()
    assert np.isnan(D[M:]).all(), "rows past M were written"
    if ldd > N:
        assert np.isnan(D[:M, N:]).all(), "padding columns were written"
    assert_fully_written(tD, M, N, "guarded D")
    check_all_rows(D, lambda r: orc.gemm("bf16", M, N, K, 1.0, A.ravel(), K, B.ravel(), N, 0.5, C.ravel(), ldd,
                                         rows=r), M, N, K, out, "bf16", "guarded D")


@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
def test_pair_beta_zero_every_output(orc, out):
    """beta = 0 on CTA pairs (C is not read; the TMA epilogue only stages D), FP16
    inputs, several units per pair with half tiles, an M tail inside a chunk."""
    M, N, K = 4000, 2560, 96
    run_gemm(orc, "f16", M, N, K, -1.25, 0.0, out)


def test_c_d_must_be_element_aligned():
    """D (or C when read) off its element alignment is rejected before any launch."""
    import linear_layer_gb300 as ll
    A = torch.zeros(64 * 64, dtype=torch.float16, device="cuda")
    raw = torch.zeros(64 * 64 * 4 + 4, dtype=torch.uint8, device="cuda")
    bad = raw[1:]  # one byte past a 4-byte boundary
    good = torch.zeros(64 * 64, dtype=torch.float32, device="cuda")
    for C, D, beta in [(None, bad, 0.0), (bad, good, 1.0)]:
        with pytest.raises(ll.LLError) as e:
            ll.gemm_f16(64, 64, 64, 1.0, A, 64, A, 64, beta, C, 64, D, 64, ll.OUT_F32)
        assert e.value.status == ll.LL_ERR_MISALIGNED
    with pytest.raises(ll.LLError) as e:
        ll.gemm_f16_noalloc(64, 64, 64, 1.0, A, 64, A, 64, 0.0, None, 64, bad, 64, ll.OUT_F32)
    assert e.value.status == ll.LL_ERR_MISALIGNED
