"""GPU parity (bit-exact z and y) of the W8A8 linear layer for a batch of tokens
(per-token activation scales, A100 page section 5.1) through the C ABI, against the
CPU oracle: token counts that fill one or several 16-token groups and ragged ones,
full-size and ragged layer shapes, padded pitches, bias and INT8 outputs."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import up

pytestmark = pytest.mark.gpu


def run_batch(orc, M, N, K, ldx=None, ldw=None, ldy=None, bias=False, out_i8=False, with_z=True):
    import linear_layer_gb300 as ll
    ldx = K if ldx is None else ldx
    ldw = K if ldw is None else ldw
    ldy = N if ldy is None else ldy
    X, s_x, W, s_W = wl.batch_w8a8_inputs(M, N, K, ldx, ldw)
    b = (np.random.default_rng(700 + N).standard_normal(N) * 2).astype(np.float32) if bias else None
    s_y = np.float32(0.05)
    z_ref, y_ref = orc.linear_w8a8(M, N, K, X, ldx, s_x, W, ldw, s_W, bias=b, out_int8=out_i8, s_y=s_y)
    ydt = torch.int8 if out_i8 else torch.float16
    tY = torch.full((M, ldy), 0, dtype=ydt, device="cuda")
    if not out_i8:
        tY.fill_(float("nan"))
    tZ = torch.full((M, N), -7, dtype=torch.int32, device="cuda") if with_z else None
    ll.linear_w8a8(M, N, K, up(X), ldx, up(s_x), up(W), ldw, up(s_W), None if b is None else up(b),
                   ll.GEMV_OUT_I8 if out_i8 else ll.GEMV_OUT_F16, torch.tensor([s_y], device="cuda"),
                   tY, ldy, tZ, N)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, word
    got = tY.cpu().numpy()[:, :N]
    if with_z:
        assert np.array_equal(tZ.cpu().numpy().astype(np.int64), z_ref)
    if out_i8:
        assert np.array_equal(got, y_ref)
    else:
        assert np.array_equal(got.view(np.uint16), y_ref.view(np.uint16))
    if ldy > N and not out_i8:
        assert np.all(np.isnan(tY.cpu().numpy()[:, N:].astype(np.float32)))  # padding untouched


@pytest.mark.parametrize("M", [2, 4, 8, 16, 32, 64])
def test_batch_full_size(orc, M):
    run_batch(orc, M, 11008, 4096)


@pytest.mark.parametrize("M", [3, 5, 9, 17, 33, 100])
def test_batch_ragged_token_counts(orc, M):
    run_batch(orc, M, 1000, 4096)


@pytest.mark.parametrize("M,N,K", [(4, 1, 16), (8, 37, 4096), (16, 300, 11008), (2, 5, 32768),
                                   (6, 129, 512), (16, 7, 48), (40, 20000, 1040), (12, 160, 40000),
                                   (64, 19457, 256), (20, 37, 4096), (32, 300, 11008), (17, 5, 48),
                                   (30, 160, 40000)])
def test_batch_shapes(orc, M, N, K):
    run_batch(orc, M, N, K)


@pytest.mark.parametrize("M", [7, 24])
def test_batch_padded_pitches(orc, M):
    run_batch(orc, M, 333, 1024, ldx=1040, ldw=1056, ldy=340)


@pytest.mark.parametrize("M", [8, 24])
def test_batch_extreme_codes_exact(orc, M):
    # x = W = -128 everywhere: every 512-K partial of the tensor-core path reaches 2^23
    # and z = K * 2^14 exactly (8 tokens: dp4a kernel; 24 tokens: tensor cores)
    import linear_layer_gb300 as ll
    N, K = 300, 8192
    X = np.full((M, K), -128, np.int8)
    W = np.full((N, K), -128, np.int8)
    W[1::2] = 127
    s_x = np.full(M, 1e-6, np.float32)
    s_W = np.full(N, 1e-3, np.float32)
    z_ref, y_ref = orc.linear_w8a8(M, N, K, X, K, s_x, W, K, s_W)
    tY = torch.empty((M, N), dtype=torch.float16, device="cuda")
    tZ = torch.empty((M, N), dtype=torch.int32, device="cuda")
    ll.linear_w8a8(M, N, K, up(X), K, up(s_x), up(W), K, up(s_W), None, ll.GEMV_OUT_F16, None, tY, N,
                   tZ, N)
    torch.cuda.synchronize()
    assert np.array_equal(tZ.cpu().numpy().astype(np.int64), z_ref)
    assert np.array_equal(tY.cpu().numpy().view(np.uint16), y_ref.view(np.uint16))


def test_batch_unaligned_falls_back_per_token(orc):
    run_batch(orc, 5, 120, 100, ldx=100, ldw=104)


@pytest.mark.parametrize("M", [12, 28])
@pytest.mark.parametrize("bias,out_i8", [(True, False), (True, True), (False, True)])
def test_batch_epilogue_variants(orc, bias, out_i8, M):
    run_batch(orc, M, 11008, 4096, bias=bias, out_i8=out_i8)


def test_batch_without_z(orc):
    run_batch(orc, 8, 500, 2048, with_z=False)


def test_batch_single_token_is_gemv(orc):
    run_batch(orc, 1, 11008, 4096, bias=True)


def test_batch_rejects_bad_arguments():
    import linear_layer_gb300 as ll
    t8 = torch.zeros(256, dtype=torch.int8, device="cuda")
    f = torch.zeros(64, dtype=torch.float32, device="cuda")
    h = torch.zeros(64, dtype=torch.float16, device="cuda")
    with pytest.raises(ll.LLError):
        ll.linear_w8a8(2, 4, 16, t8, 8, f, t8, 16, f, None, ll.GEMV_OUT_F16, None, h, 4)   # ldx < K
    with pytest.raises(ll.LLError):
        ll.linear_w8a8(2, 4, 16, t8, 16, f, t8, 16, f, None, ll.GEMV_OUT_F16, None, h, 3)  # ldy < N
    with pytest.raises(ll.LLError):
        ll.linear_w8a8(2, 4, 16, t8, 16, f, t8, 16, f, None, ll.GEMV_OUT_I8, None, t8, 4)  # no y_scale
    with pytest.raises(ll.LLError):
        ll.linear_w8a8(2, 4, 131072, t8, 131072, f, t8, 131072, f, None, ll.GEMV_OUT_F16, None, h, 4)
