"""Seeded synthetic inputs for the linear-layer hot path.

This module only draws random inputs and lays them out in memory; it holds none
of the method's arithmetic.  Both the CUDA path (tests, bench) and the CPU oracle
consume exactly the bytes produced here.

Generator: numpy ``default_rng(seed)`` (PCG64), values drawn in row-major order.
Seeds: A = 1, B = 2, C = 3, scales = 4, x = 5, s_x = 6 (the GEMM seeds 1 and 2 are the ones
the "Tensor Core" chapter's WMMA host harness uses for A and B).

Distributions (the workload shapes of the pages' linear layer):

* FP16 operands: U[-1, 1] in float64, rounded to FP16 (round to nearest even).
* BF16 operands: N(0, 1) drawn in float32, rounded to BF16 (nearest even).
* FP32 C: N(0, 1) in float32.
* int8 activations and weights: integers uniform on [-127, 127] (so -128 never occurs).
* FP32 scales: U(0.001, 0.02).
* FP8 E4M3 operands: N(0, 1) in float32, one FP32 scale per block
  s = amax(|block|) / 448 (s = 1 for an all-zero block), code = e4m3(x / s) rounded
  to nearest even; blocks are 1 x 128 for A and 128 x 128 for B.  Turning the FP32
  values into E4M3 bytes uses torch's float8_e4m3fn conversion.  E5M2 operands the
  same with amax / 57344 and torch's float8_e5m2.

Leading dimensions larger than the row width leave padding columns; they are
filled with a NaN code so that a kernel which reads padding poisons its result.
"""
import numpy as np

SEED_A, SEED_B, SEED_C, SEED_SCALE, SEED_X, SEED_SX = 1, 2, 3, 4, 5, 6

NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0, "e4m3": 0x7F}

# The workloads of the linear layer (named by what they are, with sizes): the five
# configurations of the path and the MX block-scaled FP8 GEMM of the FP8 size.
WORKLOADS = {
    "f16_gemm_256": dict(op="gemm", kind="f16", M=256, N=256, K=256, alpha=1.0, beta=0.0,
                         out="f32"),
    "bf16_gemm_4096": dict(op="gemm", kind="bf16", M=4096, N=4096, K=4096, alpha=1.0, beta=1.0,
                           out="bf16"),
    "w8a8_gemv_4096x11008": dict(op="gemv", N=11008, K=4096),
    "f16_gemm_4093x5003x2056": dict(op="gemm", kind="f16", M=4093, N=5003, K=2056, alpha=0.5,
                                    beta=-1.25, out="f32"),
    "e4m3_gemm_8192": dict(op="fp8", kind="e4m3", M=8192, N=8192, K=8192, alpha=1.0, beta=0.0,
                           out="bf16"),
    "mxf8_gemm_8192": dict(op="gemm_mx", kind="e4m3", M=8192, N=8192, K=8192, alpha=1.0, beta=0.0,
                           out="bf16"),
    "nvf4_gemm_8192": dict(op="gemm_nvf4", kind="e2m1", M=8192, N=8192, K=8192, alpha=1.0, beta=0.0,
                           out="bf16"),
}


def _pad(vals, ld, fill, dtype):
    rows, cols = vals.shape
    if ld < cols:
        raise ValueError("leading dimension smaller than the row width")
    out = np.full((rows, ld), fill, dtype=dtype)
    out[:, :cols] = vals
    return out


def f16_uniform(rows, cols, seed, ld=None):
    """FP16 bits (uint16, rows x ld) of U[-1, 1] draws."""
    ld = cols if ld is None else ld
    v = np.random.default_rng(seed).uniform(-1.0, 1.0, size=(rows, cols))
    bits = v.astype(np.float16).view(np.uint16)
    return _pad(bits, ld, NAN_BITS["f16"], np.uint16)


def bf16_normal(rows, cols, seed, ld=None):
    """BF16 bits (uint16, rows x ld) of N(0, 1) draws."""
    import torch
    ld = cols if ld is None else ld
    v = np.random.default_rng(seed).standard_normal(size=(rows, cols), dtype=np.float32)
    bits = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return _pad(bits, ld, NAN_BITS["bf16"], np.uint16)


def operand(kind, rows, cols, seed, ld=None):
    if kind == "f16":
        return f16_uniform(rows, cols, seed, ld)
    if kind == "bf16":
        return bf16_normal(rows, cols, seed, ld)
    raise ValueError(kind)


def f32_normal(rows, cols, seed, ld=None):
    ld = cols if ld is None else ld
    v = np.random.default_rng(seed).standard_normal(size=(rows, cols), dtype=np.float32)
    return _pad(v, ld, np.float32(np.nan), np.float32)


def int8_uniform(shape, seed):
    return np.random.default_rng(seed).integers(-127, 128, size=shape, dtype=np.int8)


def scales_uniform(n, seed, lo=0.001, hi=0.02):
    return np.random.default_rng(seed).uniform(lo, hi, size=n).astype(np.float32)


F8_MAX = {"e4m3": 448.0, "e5m2": 57344.0}


def _to_f8_bits(v32, fmt="e4m3"):
    import torch
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    t = torch.from_numpy(np.ascontiguousarray(v32)).to(dt)
    return t.view(torch.uint8).numpy()


def _to_e4m3_bits(v32):
    return _to_f8_bits(v32, "e4m3")


def e4m3_blockquant(rows, cols, seed, block_rows, block_cols, ld=None, fmt="e4m3"):
    """Quantise N(0, 1) float32 draws to E4M3 (or E5M2) per block of block_rows x block_cols.

    Returns (codes uint8 rows x ld, scales float32 ceil(rows/br) x ceil(cols/bc)).
    """
    ld = cols if ld is None else ld
    v = np.random.default_rng(seed).standard_normal(size=(rows, cols), dtype=np.float32)
    nbr = -(-rows // block_rows)
    nbc = -(-cols // block_cols)
    scales = np.ones((nbr, nbc), dtype=np.float32)
    q = np.empty((rows, cols), dtype=np.float32)
    for bi in range(nbr):
        r0, r1 = bi * block_rows, min(rows, (bi + 1) * block_rows)
        blk = v[r0:r1]
        for bj in range(nbc):
            c0, c1 = bj * block_cols, min(cols, (bj + 1) * block_cols)
            amax = np.float32(np.max(np.abs(blk[:, c0:c1]))) if (r1 > r0 and c1 > c0) else 0
            s = np.float32(amax) / np.float32(F8_MAX[fmt]) if amax > 0 else np.float32(1.0)
            scales[bi, bj] = s
            q[r0:r1, c0:c1] = blk[:, c0:c1] / s
    codes = _to_f8_bits(q, fmt)
    return _pad(codes, ld, NAN_BITS["e4m3"], np.uint8), scales


def e4m3_blockquant_rowblocks(rows, cols, seed, ld=None, fmt="e4m3"):
    """A operand: 1 x 128 blocks (one scale per row and 128-wide K block)."""
    ld = cols if ld is None else ld
    v = np.random.default_rng(seed).standard_normal(size=(rows, cols), dtype=np.float32)
    nbc = -(-cols // 128)
    pad = nbc * 128 - cols
    vp = np.pad(v, ((0, 0), (0, pad))) if pad else v
    blocks = vp.reshape(rows, nbc, 128)
    amax = np.max(np.abs(blocks), axis=2).astype(np.float32)
    scales = np.where(amax > 0, amax / np.float32(F8_MAX[fmt]), np.float32(1.0)).astype(np.float32)
    q = (blocks / scales[:, :, None]).reshape(rows, nbc * 128)[:, :cols]
    codes = _to_f8_bits(q.astype(np.float32), fmt)
    return _pad(codes, ld, NAN_BITS["e4m3"], np.uint8), scales


def gemm_inputs(kind, M, N, K, beta, lda=None, ldb=None, ldc=None):
    """Operands of a 16-bit GEMM workload: A (M x lda), B (K x ldb), C (M x ldc) or None."""
    A = operand(kind, M, K, SEED_A, lda)
    B = operand(kind, K, N, SEED_B, ldb)
    C = f32_normal(M, N, SEED_C, ldc) if beta != 0.0 else None
    return A, B, C


def fp8_inputs(M, N, K, beta=0.0, lda=None, ldb=None, ldc=None):
    """E4M3 operands with block scales: (A, sA, B, sB, C or None)."""
    A, sA = e4m3_blockquant_rowblocks(M, K, SEED_A, lda)
    B, sB = e4m3_blockquant(K, N, SEED_B, 128, 128, ldb)
    C = f32_normal(M, N, SEED_C, ldc) if beta != 0.0 else None
    return A, sA, B, sB, C


def batch_w8a8_inputs(M, N, K, ldx=None, ldw=None):
    """A batch of M int8 tokens for the W8A8 layer: (X int8 [M x ldx], s_x float32 [M],
    W int8 [N x ldw], s_W float32 [N]); token 0 and the weights are those of
    gemv_inputs, so the batch-1 case is the same layer."""
    ldx = K if ldx is None else ldx
    x0, _, W, s_W = gemv_inputs(N, K, ldw)
    X = np.full((M, ldx), 77, dtype=np.int8)  # padding a kernel must not read
    if M > 0:
        X[0, :K] = x0
        if M > 1:
            X[1:, :K] = int8_uniform((M - 1, K), SEED_X + 100)
    s_x = scales_uniform(M, SEED_SX)
    return X, s_x, W, s_W


def w8a16_inputs(M, N, K, ldx=None, ldw=None):
    """Weight-only layer inputs: (X BF16 codes uint16 [M x ldx], W int8 [N x ldw],
    s_W float32 [N]); X ~ N(0,1) rounded to BF16, W and s_W as gemv_inputs."""
    _, _, W, s_W = gemv_inputs(N, K, ldw)
    X = bf16_normal(M, K, SEED_X + 200, ldx)  # NaN codes in the padding
    return X, W, s_W


def gemv_inputs(N, K, ldw=None):
    """(x int8 [K], s_x float32 scalar, W int8 [N x ldw], s_W float32 [N])."""
    ldw = K if ldw is None else ldw
    x = int8_uniform(K, SEED_X)
    s_x = scales_uniform(1, SEED_SX)[0]
    W = int8_uniform((N, K), SEED_B)
    if ldw != K:
        Wp = np.full((N, ldw), 77, dtype=np.int8)  # padding a kernel must not read
        Wp[:, :K] = W
        W = Wp
    s_W = scales_uniform(N, SEED_SCALE)
    return x, s_x, W, s_W

F8_EMAX = {"e4m3": 8, "e5m2": 15}  # exponent of the largest power of two below the format's maximum


def mx_quant(rows, cols, seed, block_axis, ld=None, fmt="e4m3", spread=4):
    """OCP microscaling (MX) quantisation of seeded N(0, 1) draws, each 32-element block
    first multiplied by 2^u (u uniform in [-spread, spread]) so the block scales differ:
    32 consecutive elements along `block_axis` (1: along a row, A's K; 0: down a column,
    B's K) share the E8M0 code e = clamp(floor(log2(amax)) - emax + 127, 0, 254), and each
    element is v / 2^(e - 127) rounded to the element format (saturating at its maximum).

    Returns (codes uint8 rows x ld, scale codes uint8: rows x ceil(cols / 32) for
    block_axis 1; for block_axis 0 (B, K x N) cols x ceil(rows / 32), one row of scales per
    column of B, K blocks contiguous)."""
    ld = cols if ld is None else ld
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(size=(rows, cols), dtype=np.float32).astype(np.float64)
    if block_axis == 1:
        nb = -(-cols // 32)
        u = rng.integers(-spread, spread + 1, size=(rows, nb))
        v = v * np.ldexp(1.0, u[:, np.arange(cols) // 32])
        amax = np.zeros((rows, nb))
        for b in range(nb):
            amax[:, b] = np.max(np.abs(v[:, 32 * b:32 * b + 32]), axis=1) if cols else 0
    else:
        nb = -(-rows // 32)
        u = rng.integers(-spread, spread + 1, size=(nb, cols))
        v = v * np.ldexp(1.0, u[np.arange(rows) // 32, :])
        amax = np.zeros((nb, cols))
        for b in range(nb):
            amax[b, :] = np.max(np.abs(v[32 * b:32 * b + 32, :]), axis=0) if rows else 0
    with np.errstate(divide="ignore"):
        x = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - F8_EMAX[fmt], -127)
    codes_s = np.clip(x + 127, 0, 254).astype(np.uint8)
    scale = np.ldexp(1.0, codes_s.astype(np.int64) - 127)
    full = scale[:, np.arange(cols) // 32] if block_axis == 1 else scale[np.arange(rows) // 32, :]
    q = np.clip(v / full, -F8_MAX[fmt], F8_MAX[fmt]).astype(np.float32)
    codes = _to_f8_bits(q, fmt)
    if block_axis == 0:
        codes_s = np.ascontiguousarray(codes_s.T)
    return _pad(codes, ld, NAN_BITS["e4m3"], np.uint8), codes_s


E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def nvf4_quant(rows, cols, seed, ld=None, spread=3):
    """NVFP4 quantisation of seeded N(0, 1) draws along rows (K contiguous), each 16-element
    block first multiplied by 2^u (u uniform in [-spread, spread]): the block's UE4M3 scale is
    amax / 6 rounded to E4M3 (1 for an all-zero block; never below the smallest normal), each
    element v / scale rounded to the nearest E2M1 magnitude (ties to the smaller one).

    Returns (codes uint8 rows x ld/2 -- two per byte, element k in byte k / 2, low nibble for
    even k -- and scale codes uint8 rows x ceil(cols / 16))."""
    import torch
    ld = cols if ld is None else ld
    if ld % 2:
        raise ValueError("FP4 pitch must be even")
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(size=(rows, cols), dtype=np.float32).astype(np.float64)
    nb = -(-cols // 16)
    u = rng.integers(-spread, spread + 1, size=(rows, nb))
    v = v * np.ldexp(1.0, u[:, np.arange(cols) // 16])
    amax = np.zeros((rows, nb))
    for b in range(nb):
        amax[:, b] = np.max(np.abs(v[:, 16 * b:16 * b + 16]), axis=1) if cols else 0
    target = np.where(amax > 0, np.maximum(amax / 6.0, 2.0 ** -6), 1.0).astype(np.float32)
    sc = torch.from_numpy(target).to(torch.float8_e4m3fn)
    scodes = sc.view(torch.uint8).numpy().copy()
    svals = sc.to(torch.float64).numpy()
    q = v / svals[:, np.arange(cols) // 16]
    mag = np.abs(q)
    vals = np.array(E2M1_VALUES)
    best = np.argmin(np.abs(mag[..., None] - vals), axis=-1)  # nearest; ties to the smaller magnitude
    codes = (best | (np.signbit(q).astype(np.int64) << 3)).astype(np.uint8)
    full = np.zeros((rows, ld), dtype=np.uint8)
    full[:, :cols] = codes
    packed = (full[:, 0::2] | (full[:, 1::2] << 4)).astype(np.uint8)
    return packed, scodes
