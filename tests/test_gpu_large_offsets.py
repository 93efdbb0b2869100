"""GPU parity where element offsets pass 2^31: operands, C, D and weights sit in buffers
whose leading dimension is so large that their last rows start more than 2^31 elements
(or bytes) in, and one D holds more than 2^31 elements at a tight pitch.  The values are
the usual seeded inputs, copied into the first columns of the wide device buffers; the
oracle sees the tight host arrays.  GEMMs are compared on sampled rows that include the
last ones; the integer layers bit for bit on every output.  Each case holds 3 to 22 GB
of device memory."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import check_close, out_code, up

pytestmark = pytest.mark.gpu

WIDE = 2 ** 19 + 64  # row pitch (elements): 4096 rows of it pass 2^31 elements


def _wide(t, rows, ld):
    """Zero-filled device buffer of rows x ld elements of t's dtype, t in its first columns."""
    w = torch.zeros((rows, ld), dtype=t.dtype, device=t.device)
    w[:, :t.shape[1]].copy_(t)
    return w


def _rows(M, seed):
    rng = np.random.default_rng(seed)
    return np.array(sorted({0, 127, 128, M // 2, M - 129, M - 2, M - 1} | set(int(r) for r in rng.integers(0, M, 5))))


def _read_rows(tD, rows, N):
    return tD[torch.from_numpy(rows).to(tD.device), :N].float().cpu().numpy().astype(np.float64)


def _ok():
    import linear_layer_gb300 as ll
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, "device status %s (word %#x)" % (ll.status_string(st), word)


def test_bf16_wide_aligned_pitches(orc):
    """A, B, C, D rows 16-byte aligned (TMA operand loads, TMA epilogue), beta = 1."""
    import linear_layer_gb300 as ll
    M = N = 4096
    K = 256
    A, B, C = wl.gemm_inputs("bf16", M, N, K, 1.0)
    tA, tB, tC = _wide(up(A), M, WIDE), _wide(up(B), K, WIDE), _wide(up(C), M, WIDE)
    tD = torch.full((M, WIDE), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert ll.gemm_workspace_size(M, N, K, WIDE, WIDE, ll.IN_BF16) == 0
    ll.gemm_bf16(M, N, K, 1.0, tA, WIDE, tB, WIDE, 1.0, tC, WIDE, tD, WIDE, ll.OUT_BF16)
    _ok()
    rows = _rows(M, 1)
    ref, absab = orc.gemm("bf16", M, N, K, 1.0, A.ravel(), K, B.ravel(), N, 1.0, C.ravel(), N, rows=rows)
    check_close(_read_rows(tD, rows, N), ref, absab, K, "bf16", "bf16", what="bf16 wide pitches")
    pad = tD[torch.from_numpy(rows).cuda(), N:N + 64].float()
    assert torch.isnan(pad).all()


def test_f16_wide_unaligned_pitches(orc):
    """A with a 2-byte-aligned pitch (repacked into the workspace by a kernel reading rows
    past 2^31 elements), C and D FP32 with a pitch that is not a multiple of 16 bytes
    (transposing epilogue), alpha 0.5, beta -1.25."""
    import linear_layer_gb300 as ll
    M = N = 4096
    K = 256
    lda, ldcd = WIDE + 3, WIDE + 1
    A, B, C = wl.gemm_inputs("f16", M, N, K, -1.25)
    tA, tB, tC = _wide(up(A), M, lda), up(B), _wide(up(C), M, ldcd)
    tD = torch.full((M, ldcd), float("nan"), dtype=torch.float32, device="cuda")
    need = ll.gemm_workspace_size(M, N, K, lda, N, ll.IN_F16)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ll.gemm_f16(M, N, K, 0.5, tA, lda, tB, N, -1.25, tC, ldcd, tD, ldcd, ll.OUT_F32, workspace=ws)
    _ok()
    rows = _rows(M, 2)
    ref, absab = orc.gemm("f16", M, N, K, 0.5, A.ravel(), K, B.ravel(), N, -1.25, C.ravel(), N, rows=rows)
    check_close(_read_rows(tD, rows, N), ref, absab, K, "f32", "f16", what="f16 wide unaligned pitches")


def test_fp8_wide_pitches(orc):
    """FP8 operands whose last rows start past 2 GiB, D BF16 past 2^31 elements."""
    import linear_layer_gb300 as ll
    M = N = 4096
    K = 256
    A, sA, B, sB, _ = wl.fp8_inputs(M, N, K)
    KB, NB = sA.shape[1], sB.shape[1]
    tA, tB = _wide(up(A), M, WIDE), _wide(up(B), K, WIDE)
    tD = torch.full((M, WIDE), float("nan"), dtype=torch.bfloat16, device="cuda")
    ll.gemm_fp8_blockscaled(M, N, K, 1.0, tA, WIDE, up(sA), KB, tB, WIDE, up(sB), NB, 0.0, None, N, tD, WIDE,
                            ll.OUT_BF16)
    _ok()
    rows = _rows(M, 3)
    ref, absab = orc.gemm_fp8_blockscaled(M, N, K, 1.0, A.ravel(), K, sA.ravel(), KB, B.ravel(), N, sB.ravel(), NB,
                                          0.0, None, N, rows=rows)
    check_close(_read_rows(tD, rows, N), ref, absab, K, "bf16", "e4m3", what="fp8 wide pitches")


def test_bf16_output_past_2g_elements_tight(orc):
    """A tight D of 70000 x 32768 BF16 (2.29e9 elements)."""
    import linear_layer_gb300 as ll
    M, N, K = 70000, 32768, 64
    A, B, _ = wl.gemm_inputs("bf16", M, N, K, 0.0)
    tD = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ll.gemm_bf16(M, N, K, 1.0, up(A), K, up(B), N, 0.0, None, N, tD, N, ll.OUT_BF16)
    _ok()
    rows = _rows(M, 4)
    ref, absab = orc.gemm("bf16", M, N, K, 1.0, A.ravel(), K, B.ravel(), N, 0.0, None, N, rows=rows)
    check_close(_read_rows(tD, rows, N), ref, absab, K, "bf16", "bf16", what="bf16 70000x32768x64")


LDW = 195088  # 11008 rows of it pass 2^31 bytes; a multiple of 16


def test_gemv_wide_weight_pitch(orc):
    import linear_layer_gb300 as ll
    N, K = 11008, 4096
    x, sx, W, sW = wl.gemv_inputs(N, K)
    tW = _wide(up(W), N, LDW)
    ty = torch.full((N,), float("nan"), dtype=torch.float16, device="cuda")
    tz = torch.zeros(N, dtype=torch.int32, device="cuda")
    ll.linear_w8a8_gemv(N, K, up(x), torch.tensor([sx], device="cuda"), tW, LDW, up(sW), ty, tz)
    _ok()
    z_ref, y_ref = orc.gemv_w8a8(N, K, x, sx, W, K, sW)
    assert np.array_equal(tz.cpu().numpy().astype(np.int64), z_ref)
    assert np.array_equal(ty.cpu().numpy().view(np.uint16), y_ref.view(np.uint16))


@pytest.mark.parametrize("M", [4, 20])
def test_w8a8_tokens_wide_weight_pitch(orc, M):
    """Several tokens: the dp4a kernel (4) and the tensor-core path (20)."""
    import linear_layer_gb300 as ll
    N, K = 11008, 4096
    X, s_x, W, s_W = wl.batch_w8a8_inputs(M, N, K)
    tW = _wide(up(W), N, LDW)
    tY = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    tZ = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
    ll.linear_w8a8(M, N, K, up(X), K, up(s_x), tW, LDW, up(s_W), None, ll.GEMV_OUT_F16,
                   torch.tensor([0.05], device="cuda"), tY, N, tZ, N)
    _ok()
    z_ref, y_ref = orc.linear_w8a8(M, N, K, X, K, s_x, W, K, s_W)
    assert np.array_equal(tZ.cpu().numpy().astype(np.int64), z_ref)
    assert np.array_equal(tY.cpu().numpy().view(np.uint16), y_ref.view(np.uint16))


@pytest.mark.parametrize("M", [1, 3])
def test_w8a16_wide_weight_pitch(orc, M):
    """Weight-only layer: the one-token row kernel (1) and the column walk (3)."""
    import linear_layer_gb300 as ll
    N, K = 11008, 4096
    X, W, s_W = wl.w8a16_inputs(M, N, K, K, K)
    tW = _wide(up(W), N, LDW)
    tY = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ll.linear_w8a16(M, N, K, up(X), K, tW, LDW, up(s_W), None, ll.OUT_BF16, tY, N)
    _ok()
    ref, ab = orc.linear_w8a16(M, N, K, X, K, W, K, s_W)
    check_close(tY.float().cpu().numpy().astype(np.float64), ref, ab, K, "bf16", "bf16", what="w8a16 wide ldw")
