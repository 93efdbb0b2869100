"""Randomised GPU parity sweep of the W8A8 linear layer (1..70 tokens: batch-1 GEMV,
dp4a and tensor-core passes; bit-exact z and y) and of the weight-only INT8 x BF16
layer (tolerance bar), seeded: random shapes, aligned and unaligned K and pitches,
bias, INT8 and FP32 / BF16 / FP16 outputs."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import check_close, out_code, out_tensor, up

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed", range(24))
def test_random_w8a8(orc, seed):
    import linear_layer_gb300 as ll
    rng = np.random.default_rng(7000 + seed)
    M = int(rng.choice([1, 2, 3, 5, 8, 13, 16, 17, 24, 31, 33, 48, 70]))
    N = int(rng.integers(1, 3000))
    aligned = rng.random() < 0.7
    K = int(rng.integers(1, 300)) * 16 if aligned else int(rng.integers(1, 4000))
    ldx = K + (int(rng.choice([0, 16, 32])) if aligned else int(rng.integers(0, 9)))
    ldw = K + (int(rng.choice([0, 16, 48])) if aligned else int(rng.integers(0, 9)))
    bias = rng.random() < 0.5
    out_i8 = rng.random() < 0.3
    X, s_x, W, s_W = wl.batch_w8a8_inputs(M, N, K, ldx, ldw)
    b = (rng.standard_normal(N) * 2).astype(np.float32) if bias else None
    s_y = np.float32(0.05)
    z_ref, y_ref = orc.linear_w8a8(M, N, K, X, ldx, s_x, W, ldw, s_W, bias=b, out_int8=out_i8, s_y=s_y)
    tY = torch.zeros((M, N), dtype=torch.int8 if out_i8 else torch.float16, device="cuda")
    tZ = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
    ll.linear_w8a8(M, N, K, up(X), ldx, up(s_x), up(W), ldw, up(s_W), None if b is None else up(b),
                   ll.GEMV_OUT_I8 if out_i8 else ll.GEMV_OUT_F16, torch.tensor([s_y], device="cuda"), tY, N, tZ, N)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, word
    what = "seed %d M %d N %d K %d ldx %d ldw %d bias %s i8 %s" % (seed, M, N, K, ldx, ldw, bias, out_i8)
    assert np.array_equal(tZ.cpu().numpy().astype(np.int64), z_ref), what
    got = tY.cpu().numpy()
    assert np.array_equal(got if out_i8 else got.view(np.uint16), y_ref if out_i8 else y_ref.view(np.uint16)), what


@pytest.mark.parametrize("seed", range(16))
def test_random_w8a16(orc, seed):
    import linear_layer_gb300 as ll
    rng = np.random.default_rng(7500 + seed)
    M = int(rng.integers(1, 11))
    N = int(rng.integers(1, 3000))
    aligned = rng.random() < 0.7
    K = int(rng.integers(1, 300)) * 16 if aligned else int(rng.integers(1, 4000))
    ldx = K + (int(rng.choice([0, 8, 24])) if aligned else int(rng.integers(0, 9)))
    ldw = K + (int(rng.choice([0, 16, 48])) if aligned else int(rng.integers(0, 9)))
    out = ["f32", "bf16", "f16"][int(rng.integers(0, 3))]
    bias = rng.random() < 0.5
    X, W, s_W = wl.w8a16_inputs(M, N, K, ldx, ldw)
    b = (rng.standard_normal(N) * 2).astype(np.float32) if bias else None
    tY = out_tensor(M, N, out)
    ll.linear_w8a16(M, N, K, up(X), ldx, up(W), ldw, up(s_W), None if b is None else up(b), out_code(out), tY, N)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, word
    ref, ab = orc.linear_w8a16(M, N, K, X, ldx, W, ldw, s_W, bias=b)
    if b is not None:
        ab = ab + np.abs(b)[None, :]
    check_close(tY.float().cpu().numpy().astype(np.float64), ref, ab, K, out, "bf16",
                what="seed %d M %d N %d K %d ldx %d ldw %d %s" % (seed, M, N, K, ldx, ldw, out))
