"""Pins of the W8A8 neighbours in the oracle ("NVIDIA A100: chip to SIMT", section 5.1):
the per-token activation quantiser (symmetric, s = amax / 127, zero point 0) and the
GEMV epilogue variants (bias in the float epilogue; INT8 requantised output).

Checks: integer-valued tokens with amax 127 quantise to themselves with s = 1; sign
symmetry; all-zero tokens; the round-trip error bound |x - q s| <= s / 2; the amax
element maps to +-127; the numpy float32 sequence bit for bit; bias = 0 and no bias
agree with the plain GEMV; W = 0 gives fp16(bias); INT8 requantisation against numpy
and its clamp.
"""
import numpy as np
import pytest

import workloads as wl


def _f16(vals):
    return np.asarray(vals, dtype=np.float64).astype(np.float16)


def test_quantize_integer_token_is_identity(orc):
    rng = np.random.default_rng(401)
    x = rng.integers(-127, 128, size=(3, 50)).astype(np.float64)
    x[:, 7] = 127.0  # amax 127 in every row
    q, s = orc.quantize_per_token_f16(3, 50, _f16(x).view(np.uint16))
    assert np.all(s == 1.0)
    assert np.array_equal(q.astype(np.int64), x.astype(np.int64))


def test_quantize_symmetry_zero_rows_and_bounds(orc):
    rng = np.random.default_rng(402)
    x = _f16(rng.standard_normal((4, 300)) * 3.0)
    x[2] = 0.0
    q, s = orc.quantize_per_token_f16(4, 300, x.view(np.uint16))
    qn, sn = orc.quantize_per_token_f16(4, 300, (-x).view(np.uint16))
    assert np.array_equal(qn, -q) and np.array_equal(sn, s)
    assert s[2] == 1.0 and np.all(q[2] == 0)
    xf = x.astype(np.float64)
    for i in (0, 1, 3):
        assert np.max(np.abs(q[i])) == 127
        assert q[i][np.argmax(np.abs(xf[i]))] == np.sign(xf[i][np.argmax(np.abs(xf[i]))]) * 127
        assert np.all(np.abs(xf[i] - q[i] * float(s[i])) <= 0.5 * float(s[i]) * (1 + 1e-6))


def test_quantize_matches_numpy_float32_sequence(orc):
    rng = np.random.default_rng(403)
    x = _f16(rng.standard_normal((5, 4096)))
    q, s = orc.quantize_per_token_f16(5, 4096, x.view(np.uint16))
    xf = x.astype(np.float32)
    amax = np.max(np.abs(xf), axis=1)
    sn = (amax / np.float32(127.0)).astype(np.float32)
    qn = np.clip(np.rint(xf / sn[:, None]), -127, 127).astype(np.int8)
    assert np.array_equal(s, sn)
    assert np.array_equal(q, qn)


def test_quantize_padded_pitch(orc):
    x = _f16(np.random.default_rng(404).standard_normal((2, 40)))
    xp = np.full((2, 48), 0x7C00, np.uint16)  # +inf in the padding must not be read
    xp[:, :40] = x.view(np.uint16)
    q1, s1 = orc.quantize_per_token_f16(2, 40, x.view(np.uint16))
    q2, s2 = orc.quantize_per_token_f16(2, 40, xp, ldx=48)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


def test_gemv_ex_without_variants_is_plain_gemv(orc):
    N, K = 70, 512
    x, sx, W, sW = wl.gemv_inputs(N, K)
    z0, y0 = orc.gemv_w8a8(N, K, x, sx, W, K, sW)
    z1, y1 = orc.gemv_w8a8_ex(N, K, x, sx, W, K, sW)
    z2, y2 = orc.gemv_w8a8_ex(N, K, x, sx, W, K, sW, bias=np.zeros(N, np.float32))
    assert np.array_equal(z0, z1) and np.array_equal(y0.view(np.uint16), y1.view(np.uint16))
    assert np.array_equal(y0.view(np.uint16), y2.view(np.uint16))


def test_gemv_ex_bias_only(orc):
    N, K = 9, 64
    bias = np.random.default_rng(405).standard_normal(N).astype(np.float32)
    _, y = orc.gemv_w8a8_ex(N, K, np.ones(K, np.int8), 0.01, np.zeros((N, K), np.int8), K,
                            np.full(N, 0.5, np.float32), bias=bias)
    assert np.array_equal(y.view(np.uint16), bias.astype(np.float16).view(np.uint16))


def test_gemv_ex_bias_and_int8_against_numpy(orc):
    N, K = 300, 4096
    x, sx, W, sW = wl.gemv_inputs(N, K)
    bias = (np.random.default_rng(406).standard_normal(N) * 4).astype(np.float32)
    zn = W.astype(np.int64) @ x.astype(np.int64)
    v = (zn.astype(np.float32) * np.float32(sx)) * sW + bias
    z, y16 = orc.gemv_w8a8_ex(N, K, x, sx, W, K, sW, bias=bias)
    assert np.array_equal(z, zn)
    assert np.array_equal(y16.view(np.uint16), v.astype(np.float16).view(np.uint16))
    s_y = np.float32(0.05)
    _, y8 = orc.gemv_w8a8_ex(N, K, x, sx, W, K, sW, bias=bias, out_int8=True, s_y=s_y)
    assert np.array_equal(y8, np.clip(np.rint(v / s_y), -127, 127).astype(np.int8))
    assert np.any(np.abs(y8) == 127)  # the clamp is exercised


def test_gemv_ex_int8_identity_scale(orc):
    # s_x = s_W = s_y = 1 and small z: the requantised output is z itself
    N, K = 5, 16
    x = np.ones(K, np.int8)
    W = np.zeros((N, K), np.int8)
    W[:, 0] = np.array([-3, -1, 0, 2, 7], np.int8)
    _, y8 = orc.gemv_w8a8_ex(N, K, x, 1.0, W, K, np.ones(N, np.float32), out_int8=True, s_y=1.0)
    assert list(y8) == [-3, -1, 0, 2, 7]


# ------------------------------------------------------- several tokens (per-token s_x)


def test_batch_against_numpy(orc):
    # z = X W^T exactly; y in the FP32 order of section 5.2 with each token's own s_x
    M, N, K = 6, 130, 1000
    X, s_x, W, s_W = wl.batch_w8a8_inputs(M, N, K, ldx=1008, ldw=1008)
    bias = (np.random.default_rng(407).standard_normal(N) * 2).astype(np.float32)
    z, y = orc.linear_w8a8(M, N, K, X, 1008, s_x, W, 1008, s_W, bias=bias)
    zn = X[:, :K].astype(np.int64) @ W[:, :K].astype(np.int64).T
    assert np.array_equal(z, zn)
    v = (zn.astype(np.float32) * s_x[:, None]) * s_W[None, :] + bias[None, :]
    assert np.array_equal(y.view(np.uint16), v.astype(np.float16).view(np.uint16))


def test_batch_token_scale_is_per_row(orc):
    # a distinct power-of-two s_x per token scales only that token's row, exactly; a
    # transposed (per-channel) use of s_x would fail this
    M, N, K = 4, 9, 64
    X = np.ones((M, K), np.int8)
    W = np.zeros((N, K), np.int8)
    W[:, 0] = np.arange(1, N + 1)
    s_x = np.array([1.0, 2.0, 0.5, 4.0], np.float32)
    _, y = orc.linear_w8a8(M, N, K, X, K, s_x, W, K, np.ones(N, np.float32))
    for m in range(M):
        assert np.array_equal(y[m].astype(np.float64), s_x[m] * np.arange(1, N + 1))


def test_batch_int8_output_and_single_token_reduction(orc):
    M, N, K = 3, 200, 4096
    X, s_x, W, s_W = wl.batch_w8a8_inputs(M, N, K)
    z8, y8 = orc.linear_w8a8(M, N, K, X, K, s_x, W, K, s_W, out_int8=True, s_y=0.05)
    v = (z8.astype(np.float32) * s_x[:, None]) * s_W[None, :]
    assert np.array_equal(y8, np.clip(np.rint(v / np.float32(0.05)), -127, 127).astype(np.int8))
    # token 0 of the batch is the batch-1 workload: the same z as the GEMV oracle
    x0, sx0, _, _ = wl.gemv_inputs(N, K)
    z1, _ = orc.gemv_w8a8(N, K, x0, sx0, W, K, s_W)
    assert np.array_equal(z8[0], z1)


# ------------------------------------------------- weight-only INT8 (BF16 activation)


def _bf16(v):
    import torch
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_w8a16_against_numpy(orc):
    M, N, K = 3, 70, 500
    X, W, s_W = wl.w8a16_inputs(M, N, K, ldx=512, ldw=512)
    bias = (np.random.default_rng(408).standard_normal(N) * 3).astype(np.float32)
    y, ab = orc.linear_w8a16(M, N, K, X, 512, W, 512, s_W, bias=bias)
    import torch
    xd = torch.from_numpy(X[:, :K].view(np.int16)).view(torch.bfloat16).double().numpy()
    ref = (xd @ W[:, :K].astype(np.float64).T) * s_W.astype(np.float64)[None, :] + bias[None, :]
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-12)
    assert np.allclose(ab, np.abs(xd) @ np.abs(W[:, :K].astype(np.float64)).T * s_W[None, :])


def test_w8a16_exact_small_integers(orc):
    # integer activations, power-of-two scales: the result is exact and hand-checkable
    X = _bf16([[1, 2, -3, 4], [0, 0, 0, 5]])
    W = np.array([[1, 1, 1, 1], [2, -1, 0, 3]], np.int8)
    s_W = np.array([0.5, 4.0], np.float32)
    y, _ = orc.linear_w8a16(2, 2, 4, X, 4, W, 4, s_W)
    assert y.tolist() == [[0.5 * 4, 4.0 * (2 - 2 + 0 + 12)], [0.5 * 5, 4.0 * 15]]


def test_w8a16_scale_is_per_output_channel(orc):
    # a transposed (per-token) use of s_W would fail
    X = _bf16(np.ones((3, 8)))
    W = np.ones((5, 8), np.int8)
    s_W = np.array([1, 2, 4, 8, 16], np.float32)
    y, _ = orc.linear_w8a16(3, 5, 8, X, 8, W, 8, s_W, bias=np.full(5, 0.25, np.float32))
    assert np.array_equal(y, np.tile(8.0 * s_W + 0.25, (3, 1)))
