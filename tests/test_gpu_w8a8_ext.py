"""GPU parity (bit-exact) of the W8A8 neighbours through the C ABI: the per-token
activation quantiser, the GEMV epilogue variants (bias, INT8 requantisation) and the
FP16-activation GEMV with the quantiser fused in, against the CPU oracle."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import up

pytestmark = pytest.mark.gpu


def _h(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to("cuda").view(torch.float16)


@pytest.mark.parametrize("M,K,ldx", [(5, 4096, 4096), (3, 100, 104), (1, 1, 1), (8, 11008, 11008),
                                     (2, 70000, 70000)])
def test_quantize_per_token_bit_exact(orc, M, K, ldx):
    import linear_layer_gb300 as ll
    rng = np.random.default_rng(500 + K)
    x = np.full((M, ldx), 0x7C00, np.uint16)  # +inf padding must not be read
    x[:, :K] = (rng.standard_normal((M, K)) * 2).astype(np.float16).view(np.uint16)
    if M > 1:
        x[1, :K] = 0  # an all-zero token
    q = torch.full((M, K), 99, dtype=torch.int8, device="cuda")
    s = torch.zeros(M, dtype=torch.float32, device="cuda")
    ll.quantize_per_token_f16(M, K, _h(x), ldx, q, K, s)
    torch.cuda.synchronize()
    q_ref, s_ref = orc.quantize_per_token_f16(M, K, x, ldx)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


def _run_ex(orc, N, K, bias, out_i8, ldw=None, fused=False, x_off=0):
    import linear_layer_gb300 as ll
    ldw = K if ldw is None else ldw
    _, _, W, sW = wl.gemv_inputs(N, K, ldw)
    rng = np.random.default_rng(600 + N)
    xh = (rng.standard_normal(K) * 3).astype(np.float16)
    xq_ref, sx_ref = orc.quantize_per_token_f16(1, K, xh.view(np.uint16).reshape(1, K))
    xq_ref, sx_ref = xq_ref[0], sx_ref[0]
    b = (rng.standard_normal(N) * 2).astype(np.float32) if bias else None
    s_y = np.float32(0.04)
    z_ref, y_ref = orc.gemv_w8a8_ex(N, K, xq_ref, sx_ref, W, ldw, sW, bias=b, out_int8=out_i8, s_y=s_y)
    ty = torch.zeros(N, dtype=torch.int8 if out_i8 else torch.float16, device="cuda")
    tz = torch.zeros(N, dtype=torch.int32, device="cuda")
    tW, tsW = up(W), up(sW)
    tb = None if b is None else up(b)
    tsy = torch.tensor([s_y], device="cuda")
    yt = ll.GEMV_OUT_I8 if out_i8 else ll.GEMV_OUT_F16
    if fused:
        buf = torch.zeros(K + 8, dtype=torch.float16, device="cuda")
        buf[x_off // 2:x_off // 2 + K] = torch.from_numpy(xh).cuda()
        xq = torch.zeros(K, dtype=torch.int8, device="cuda")
        xs = torch.zeros(1, dtype=torch.float32, device="cuda")
        ll.linear_f16_w8a8_gemv(N, K, buf.data_ptr() + x_off, xq, xs, tW, ldw, tsW, tb, yt, tsy, ty, tz)
        torch.cuda.synchronize()
        assert np.array_equal(xq.cpu().numpy(), xq_ref)
        assert xs.item() == float(sx_ref)
    else:
        ll.linear_w8a8_gemv_ex(N, K, up(xq_ref), torch.tensor([sx_ref], device="cuda"), tW, ldw, tsW, tb,
                               yt, tsy, ty, tz)
        torch.cuda.synchronize()
    assert np.array_equal(tz.cpu().numpy().astype(np.int64), z_ref)
    got = ty.cpu().numpy()
    if out_i8:
        assert np.array_equal(got, y_ref)
    else:
        assert np.array_equal(got.view(np.uint16), y_ref.view(np.uint16))


@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("out_i8", [False, True])
def test_gemv_ex_full_size(orc, bias, out_i8):
    _run_ex(orc, 11008, 4096, bias, out_i8)


@pytest.mark.parametrize("N,K,ldw", [(33, 100, 112), (64, 4096, 4112), (7, 16, 16)])
def test_gemv_ex_shapes(orc, N, K, ldw):
    _run_ex(orc, N, K, True, True, ldw=ldw)


@pytest.mark.parametrize("bias,out_i8", [(False, False), (True, False), (True, True)])
def test_fused_f16_activation_full_size(orc, bias, out_i8):
    _run_ex(orc, 11008, 4096, bias, out_i8, fused=True)


def test_fused_unaligned_activation_falls_back(orc):
    # x starts 2 bytes past a 16-byte boundary: quantiser kernel + plain GEMV, same bits
    _run_ex(orc, 300, 4096, True, False, fused=True, x_off=2)


def test_fused_odd_k(orc):
    _run_ex(orc, 50, 200, True, True, ldw=208, fused=True)


def test_ex_rejects_bad_arguments():
    import linear_layer_gb300 as ll
    t8 = torch.zeros(64, dtype=torch.int8, device="cuda")
    f = torch.zeros(64, dtype=torch.float32, device="cuda")
    with pytest.raises(ll.LLError):
        ll.linear_w8a8_gemv_ex(4, 16, t8, f, t8, 16, f, None, 7, None, f)   # unknown y_type
    with pytest.raises(ll.LLError):
        ll.linear_w8a8_gemv_ex(4, 16, t8, f, t8, 16, f, None, ll.GEMV_OUT_I8, None, t8)  # no y_scale
    with pytest.raises(ll.LLError):
        ll.quantize_per_token_f16(2, 16, f, 8, t8, 16, f)  # ldx < K


def test_int8_layer_output_as_next_weights_under_the_ordering_rule(orc):
    """The ordering rule for weights (programmatic dependent launch): a W8A8 layer reads W
    before it waits for the work before it, so W may not be an output of a library call
    that could still be running.  Here the INT8 output of ll_linear_w8a8 becomes the
    weight matrix of the next GEMV, with a kernel that does not come from the library
    in between, as the rule asks; the GEMV must see the finished matrix, bit for bit,
    and the result must equal the same GEMV on a copy that was synchronised first."""
    import linear_layer_gb300 as ll
    M, N, K = 48, 4096, 1024                 # producer: 48 tokens x 4096 channels, K 1024
    X, sx, W, sW = wl.batch_w8a8_inputs(M, N, K)
    s_y = np.float32(0.5)
    _, Yq_ref = orc.linear_w8a8(M, N, K, X, K, sx, W, K, sW, out_int8=True, s_y=s_y)
    x2 = wl.int8_uniform((N,), 77)            # consumer: W' = Y (48 x 4096), x' of 4096
    s_w2 = wl.scales_uniform(M, 78)
    z_ref, y_ref = orc.gemv_w8a8(M, N, x2, np.float32(0.01), Yq_ref, N, s_w2)
    stream = torch.cuda.Stream()
    tX, tsx, tW, tsW = up(X), up(sx), up(W), up(sW)
    tsy = torch.tensor([s_y], device="cuda")
    tx2, tsx2, tsw2 = up(x2), torch.tensor([0.01], dtype=torch.float32, device="cuda"), up(s_w2)
    other = torch.zeros(1 << 20, device="cuda")
    for rep in range(3):
        Y = torch.full((M, N), 99, dtype=torch.int8, device="cuda")
        y = torch.full((M,), float("nan"), dtype=torch.float16, device="cuda")
        z = torch.zeros(M, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        ll.linear_w8a8(M, N, K, tX, K, tsx, tW, K, tsW, None, ll.GEMV_OUT_I8, tsy, Y, N, stream=stream)
        with torch.cuda.stream(stream):
            other.add_(1.0)                   # a kernel that does not come from this library
        ll.linear_w8a8_gemv(M, N, tx2, tsx2, Y, N, tsw2, y, z, stream=stream)
        stream.synchronize()
        assert np.array_equal(Y.cpu().numpy(), Yq_ref), rep
        assert np.array_equal(z.cpu().numpy().astype(np.int64), z_ref), rep
        assert np.array_equal(y.cpu().numpy().view(np.uint16), y_ref.view(np.uint16)), rep
