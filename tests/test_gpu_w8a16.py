"""GPU parity of the weight-only INT8 linear layer with BF16 activations (tolerance bar
of the 16-bit GEMMs, FP32 accumulation) through the C ABI, against the CPU oracle;
determinism run to run."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import check_close, out_code, out_tensor, up

pytestmark = pytest.mark.gpu


def run_wo(orc, M, N, K, out="bf16", ldx=None, ldw=None, ldy=None, bias=False, rows=None):
    import linear_layer_gb300 as ll
    ldx = K if ldx is None else ldx
    ldw = K if ldw is None else ldw
    ldy = N if ldy is None else ldy
    X, W, s_W = wl.w8a16_inputs(M, N, K, ldx, ldw)
    b = (np.random.default_rng(800 + N).standard_normal(N) * 2).astype(np.float32) if bias else None
    tY = out_tensor(M, ldy, out)
    ll.linear_w8a16(M, N, K, up(X), ldx, up(W), ldw, up(s_W), None if b is None else up(b), out_code(out),
                    tY, ldy)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, word
    got = tY.float().cpu().numpy().astype(np.float64)
    ref, ab = orc.linear_w8a16(M, N, K, X, ldx, W, ldw, s_W, bias=b)
    if ab.size:
        ab = ab + (np.abs(b)[None, :] if b is not None else 0.0)
    check_close(got[:, :N], ref, ab, K, out, "bf16", what="w8a16 %dx%dx%d %s" % (M, N, K, out))
    if ldy > N:
        assert np.all(np.isnan(got[:, N:]))
    return tY


@pytest.mark.parametrize("M", [1, 2, 3, 4, 7])
def test_w8a16_full_size(orc, M):
    run_wo(orc, M, 11008, 4096)


@pytest.mark.parametrize("out", ["f32", "f16"])
def test_w8a16_outputs_and_bias(orc, out):
    run_wo(orc, 3, 1000, 4096, out=out, bias=True)


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (2, 37, 4096), (4, 300, 11008), (1, 5, 32768),
                                   (5, 129, 512), (4, 7, 48), (2, 64, 131072)])
def test_w8a16_shapes(orc, M, N, K):
    run_wo(orc, M, N, K)


def test_w8a16_padded_pitches(orc):
    run_wo(orc, 3, 333, 1024, ldx=1032, ldw=1040, ldy=340)


def test_w8a16_unaligned_plain_kernel(orc):
    run_wo(orc, 2, 120, 100, ldx=100, ldw=101, bias=True)


def test_w8a16_deterministic():
    import linear_layer_gb300 as ll
    M, N, K = 4, 11008, 4096
    X, W, s_W = wl.w8a16_inputs(M, N, K)
    tX, tW, ts = up(X), up(W), up(s_W)
    outs = []
    for _ in range(3):
        tY = torch.empty((M, N), dtype=torch.float32, device="cuda")
        ll.linear_w8a16(M, N, K, tX, K, tW, K, ts, None, ll.OUT_F32, tY, N)
        outs.append(tY.cpu())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_w8a16_rejects_bad_arguments():
    import linear_layer_gb300 as ll
    t8 = torch.zeros(64, dtype=torch.int8, device="cuda")
    f = torch.zeros(64, dtype=torch.float32, device="cuda")
    with pytest.raises(ll.LLError):
        ll.linear_w8a16(2, 4, 16, f, 8, t8, 16, f, None, ll.OUT_BF16, f, 4)   # ldx < K
    with pytest.raises(ll.LLError):
        ll.linear_w8a16(2, 4, 16, f, 16, t8, 16, f, None, 9, f, 4)             # unknown y_type
