"""CPU oracle for the linear-layer hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (``linear_layer_gb300``)
never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, double / int64 accumulation);
this module only marshals numpy arrays into it through ctypes.

Functions and the passages they follow:

* ``decode_f16`` / ``decode_bf16`` / ``decode_e4m3`` -- "Tensor Core" chapter,
  table "精度：FP16、BF16、TF32、FP8" (bit splits 1/5/10, 1/8/7, 1/4/3).
* ``gemm`` -- same chapter, section "Tensor Core 做什么": D = A x B + C with
  low-precision inputs and a wide accumulator; here alpha*A*B + beta*C in double.
* ``gemm_fp8_blockscaled`` -- same chapter, "精度" section: FP8 needs scaling
  factors per tensor, row or block; 1x128 blocks of A, 128x128 blocks of B.
* ``decode_e5m2`` / ``gemm_f8_blockscaled_mixed`` -- "Tensor Core" chapter, table
  "精度": FP8 E5M2 1/5/2 (wider range, used for gradients) beside E4M3.
* ``decode_ue8m0`` / ``gemm_mx_f8`` -- "Tensor Core" chapter, the table of formats per
  generation (Blackwell: block-scaled formats such as MXFP4 / NVFP4): OCP microscaling,
  one E8M0 scale 2^(e-127) shared by 32 consecutive K elements of a row of A or a
  column of B, scales stored K-block-contiguous per row of A / column of B (the pages
  name the formats only).
* ``decode_e2m1`` / ``decode_ue4m3`` / ``gemm_nvf4`` -- the same table: FP4 E2M1 elements
  in blocks of 16 along K sharing one UE4M3 scale (NVFP4), B given K-major.
* ``gemv_w8a8`` -- "NVIDIA A100: chip to SIMT", sections 5.1-5.2: int8 x int8
  summed exactly, then y = fp16(float(z) * s_x * s_W[o]).
* ``quantize_per_token_f16`` -- same page, 5.1: the activation is quantised per token
  at run time (symmetric, s = amax / 127, zero point 0).
* ``gemv_w8a8_ex`` -- same page, 5.1: optional bias in the float epilogue, or an INT8
  requantised output for a next layer that takes INT8.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_decode_f16.restype = ctypes.c_double
        L.orc_decode_f16.argtypes = [ctypes.c_uint16]
        L.orc_decode_bf16.restype = ctypes.c_double
        L.orc_decode_bf16.argtypes = [ctypes.c_uint16]
        L.orc_decode_e4m3.restype = ctypes.c_double
        L.orc_decode_e4m3.argtypes = [ctypes.c_uint8]
        L.orc_decode_e5m2.restype = ctypes.c_double
        L.orc_decode_e5m2.argtypes = [ctypes.c_uint8]
        L.orc_decode_e2m1.restype = ctypes.c_double
        L.orc_decode_e2m1.argtypes = [ctypes.c_uint8]
        L.orc_decode_ue4m3.restype = ctypes.c_double
        L.orc_decode_ue4m3.argtypes = [ctypes.c_uint8]
        L.orc_decode_ue8m0.restype = ctypes.c_double
        L.orc_decode_ue8m0.argtypes = [ctypes.c_uint8]
        L.orc_encode_f16_rn.restype = ctypes.c_uint16
        L.orc_encode_f16_rn.argtypes = [ctypes.c_double]
        vp = ctypes.c_void_p
        i64 = ctypes.c_int64
        L.orc_gemm.restype = ctypes.c_int
        L.orc_gemm.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               ctypes.c_double, vp, i64, vp, i64, ctypes.c_double, vp, i64,
                               vp, ctypes.c_int, vp, vp]
        L.orc_gemm_fp8_blockscaled.restype = ctypes.c_int
        L.orc_gemm_fp8_blockscaled.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_double, vp, i64, vp, i64, vp, i64,
                                               vp, i64, ctypes.c_double, vp, i64, vp,
                                               ctypes.c_int, vp, vp]
        L.orc_gemm_f8_blockscaled_mixed.restype = ctypes.c_int
        L.orc_gemm_f8_blockscaled_mixed.argtypes = [ctypes.c_int, ctypes.c_int] + \
            L.orc_gemm_fp8_blockscaled.argtypes
        L.orc_gemm_mx_f8.restype = ctypes.c_int
        L.orc_gemm_mx_f8.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_double, vp, i64, vp, i64, vp, i64, vp, i64, ctypes.c_double, vp,
                                     i64, vp, ctypes.c_int, vp, vp]
        L.orc_gemm_nvf4.restype = ctypes.c_int
        L.orc_gemm_nvf4.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, vp, i64, vp, i64,
                                    vp, i64, vp, i64, ctypes.c_double, vp, i64, vp, ctypes.c_int, vp, vp]
        L.orc_quantize_per_token_f16.restype = ctypes.c_int
        L.orc_quantize_per_token_f16.argtypes = [ctypes.c_int, ctypes.c_int, vp, i64, vp, i64, vp]
        L.orc_gemv_w8a8_ex.restype = ctypes.c_int
        L.orc_linear_w8a16.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, i64, vp, i64, vp, vp,
                                       vp, vp]
        L.orc_linear_w8a8.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, i64, vp, vp, i64,
                                      vp, vp, ctypes.c_int, ctypes.c_float, vp, vp, vp, i64]
        L.orc_gemv_w8a8_ex.argtypes = [ctypes.c_int, ctypes.c_int, vp, ctypes.c_float, vp, i64, vp,
                                       vp, ctypes.c_int, ctypes.c_float, vp, vp, vp]
        L.orc_gemv_w8a8.restype = ctypes.c_int
        L.orc_gemv_w8a8.argtypes = [ctypes.c_int, ctypes.c_int, vp, ctypes.c_float, vp, i64,
                                    vp, vp, vp]
        _lib = L
    return _lib


KIND = {"f16": 0, "bf16": 1, "e4m3": 2}


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def decode_f16(bits: int) -> float:
    return lib().orc_decode_f16(int(bits) & 0xFFFF)


def decode_bf16(bits: int) -> float:
    return lib().orc_decode_bf16(int(bits) & 0xFFFF)


def decode_e4m3(bits: int) -> float:
    return lib().orc_decode_e4m3(int(bits) & 0xFF)


def decode_e5m2(bits: int) -> float:
    return lib().orc_decode_e5m2(int(bits) & 0xFF)


def decode_e2m1(bits: int) -> float:
    return lib().orc_decode_e2m1(int(bits) & 0xF)


def decode_ue4m3(bits: int) -> float:
    return lib().orc_decode_ue4m3(int(bits) & 0xFF)


def decode_ue8m0(bits: int) -> float:
    return lib().orc_decode_ue8m0(int(bits) & 0xFF)


def encode_f16_rn(v: float) -> int:
    return lib().orc_encode_f16_rn(float(v))


def _rows(M, rows):
    if rows is None:
        rows = np.arange(M, dtype=np.int32)
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int32))


def gemm(kind, M, N, K, alpha, A, lda, B, ldb, beta=0.0, C=None, ldc=0, rows=None,
         want_absab=True):
    """Reference D (double, len(rows) x N) and sum_k |A||B| for the selected rows.

    ``A``/``B`` are flat numpy arrays holding the raw element bits (uint16 for
    f16/bf16, uint8 for e4m3) with leading dimensions ``lda``/``ldb``; ``C`` is
    float32 with ``ldc`` and is not read when ``beta == 0``.
    """
    rows = _rows(M, rows)
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    C = None if C is None else np.ascontiguousarray(C, dtype=np.float32)
    D = np.zeros((len(rows), N), dtype=np.float64)
    S = np.zeros((len(rows), N), dtype=np.float64) if want_absab else None
    rc = lib().orc_gemm(KIND[kind], M, N, K, float(alpha), _ptr(A), lda, _ptr(B), ldb,
                        float(beta), _ptr(C), ldc, _ptr(rows), len(rows), _ptr(D), _ptr(S))
    if rc != 0:
        raise ValueError("orc_gemm failed with code %d" % rc)
    return D, S


def gemm_fp8_blockscaled(M, N, K, alpha, A, lda, sA, ld_sa, B, ldb, sB, ld_sb, beta=0.0,
                         C=None, ldc=0, rows=None, want_absab=True):
    rows = _rows(M, rows)
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    sA = np.ascontiguousarray(sA, dtype=np.float32)
    sB = np.ascontiguousarray(sB, dtype=np.float32)
    C = None if C is None else np.ascontiguousarray(C, dtype=np.float32)
    D = np.zeros((len(rows), N), dtype=np.float64)
    S = np.zeros((len(rows), N), dtype=np.float64) if want_absab else None
    rc = lib().orc_gemm_fp8_blockscaled(M, N, K, float(alpha), _ptr(A), lda, _ptr(sA), ld_sa,
                                        _ptr(B), ldb, _ptr(sB), ld_sb, float(beta), _ptr(C),
                                        ldc, _ptr(rows), len(rows), _ptr(D), _ptr(S))
    if rc != 0:
        raise ValueError("orc_gemm_fp8_blockscaled failed with code %d" % rc)
    return D, S


F8 = {"e4m3": 0, "e5m2": 1}


def gemm_f8_blockscaled_mixed(a_fmt, b_fmt, M, N, K, alpha, A, lda, sA, ld_sa, B, ldb, sB, ld_sb,
                              beta=0.0, C=None, ldc=0, rows=None, want_absab=True):
    """Block-scaled 8-bit GEMM with per-operand formats ("e4m3" / "e5m2")."""
    rows = _rows(M, rows)
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    sA = np.ascontiguousarray(sA, dtype=np.float32)
    sB = np.ascontiguousarray(sB, dtype=np.float32)
    C = None if C is None else np.ascontiguousarray(C, dtype=np.float32)
    D = np.zeros((len(rows), N), dtype=np.float64)
    S = np.zeros((len(rows), N), dtype=np.float64) if want_absab else None
    rc = lib().orc_gemm_f8_blockscaled_mixed(F8[a_fmt], F8[b_fmt], M, N, K, float(alpha), _ptr(A),
                                             lda, _ptr(sA), ld_sa, _ptr(B), ldb, _ptr(sB), ld_sb,
                                             float(beta), _ptr(C), ldc, _ptr(rows), len(rows),
                                             _ptr(D), _ptr(S))
    if rc != 0:
        raise ValueError("orc_gemm_f8_blockscaled_mixed failed with code %d" % rc)
    return D, S


def gemm_mx_f8(a_fmt, b_fmt, M, N, K, alpha, A, lda, SA, ld_sa, B, ldb, SB, ld_sb, beta=0.0, C=None, ldc=0,
               rows=None, want_absab=True):
    """MX block-scaled 8-bit GEMM: element formats "e4m3" / "e5m2", E8M0 scale codes SA
    (M x ld_sa, one per row of A and 32-wide K block) and SB (N x ld_sb, one per column of B
    and K block).  Returns (D double [len(rows), N], absab)."""
    rows = _rows(M, rows)
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    SA = np.ascontiguousarray(SA, dtype=np.uint8)
    SB = np.ascontiguousarray(SB, dtype=np.uint8)
    C = None if C is None else np.ascontiguousarray(C, dtype=np.float32)
    D = np.zeros((len(rows), N), dtype=np.float64)
    S = np.zeros((len(rows), N), dtype=np.float64) if want_absab else None
    rc = lib().orc_gemm_mx_f8(F8[a_fmt], F8[b_fmt], M, N, K, float(alpha), _ptr(A), lda, _ptr(SA), ld_sa,
                              _ptr(B), ldb, _ptr(SB), ld_sb, float(beta), _ptr(C), ldc, _ptr(rows), len(rows),
                              _ptr(D), _ptr(S))
    if rc != 0:
        raise ValueError("orc_gemm_mx_f8 failed with code %d" % rc)
    return D, S


def gemm_nvf4(M, N, K, alpha, A, lda, SA, ld_sa, Bt, ldbt, SB, ld_sb, beta=0.0, C=None, ldc=0, rows=None,
              want_absab=True):
    """NVFP4 GEMM: E2M1 codes packed two per byte (A M x lda elements, Bt N x ldbt elements,
    Bt row j = column j of B), UE4M3 scale codes per 16 K elements (SA M x ld_sa, SB N x
    ld_sb).  Returns (D double [len(rows), N], absab)."""
    rows = _rows(M, rows)
    A = np.ascontiguousarray(A, dtype=np.uint8)
    Bt = np.ascontiguousarray(Bt, dtype=np.uint8)
    SA = np.ascontiguousarray(SA, dtype=np.uint8)
    SB = np.ascontiguousarray(SB, dtype=np.uint8)
    C = None if C is None else np.ascontiguousarray(C, dtype=np.float32)
    D = np.zeros((len(rows), N), dtype=np.float64)
    S = np.zeros((len(rows), N), dtype=np.float64) if want_absab else None
    rc = lib().orc_gemm_nvf4(M, N, K, float(alpha), _ptr(A), lda, _ptr(SA), ld_sa, _ptr(Bt), ldbt, _ptr(SB), ld_sb,
                             float(beta), _ptr(C), ldc, _ptr(rows), len(rows), _ptr(D), _ptr(S))
    if rc != 0:
        raise ValueError("orc_gemm_nvf4 failed with code %d" % rc)
    return D, S


def gemv_w8a8(N, K, x, s_x, W, ldw, s_W):
    """Return (z int64 [N], y float16 [N]) for the batch-1 W8A8 linear layer."""
    x = np.ascontiguousarray(x, dtype=np.int8)
    W = np.ascontiguousarray(W, dtype=np.int8)
    s_W = np.ascontiguousarray(s_W, dtype=np.float32)
    z = np.zeros(N, dtype=np.int64)
    y = np.zeros(N, dtype=np.uint16)
    rc = lib().orc_gemv_w8a8(N, K, _ptr(x), float(np.float32(s_x)), _ptr(W), ldw, _ptr(s_W),
                             _ptr(z), _ptr(y))
    if rc == 5:
        raise OverflowError("W8A8 dot product exceeds the INT32 range")
    if rc != 0:
        raise ValueError("orc_gemv_w8a8 failed with code %d" % rc)
    return z, y.view(np.float16)


def quantize_per_token_f16(M, K, x_bits, ldx=None):
    """(q int8 M x K, s float32 [M]) from FP16 bits x (M x ldx)."""
    ldx = K if ldx is None else ldx
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    q = np.zeros((M, K), dtype=np.int8)
    s = np.zeros(M, dtype=np.float32)
    rc = lib().orc_quantize_per_token_f16(M, K, _ptr(x), ldx, _ptr(q), K, _ptr(s))
    if rc != 0:
        raise ValueError("orc_quantize_per_token_f16 failed with code %d" % rc)
    return q, s


def gemv_w8a8_ex(N, K, x, s_x, W, ldw, s_W, bias=None, out_int8=False, s_y=1.0):
    """(z int64 [N], y) with y FP16 [N] or int8 [N] (out_int8)."""
    x = np.ascontiguousarray(x, dtype=np.int8)
    W = np.ascontiguousarray(W, dtype=np.int8)
    s_W = np.ascontiguousarray(s_W, dtype=np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    z = np.zeros(N, dtype=np.int64)
    y16 = np.zeros(N, dtype=np.uint16)
    y8 = np.zeros(N, dtype=np.int8)
    rc = lib().orc_gemv_w8a8_ex(N, K, _ptr(x), float(np.float32(s_x)), _ptr(W), ldw, _ptr(s_W),
                                _ptr(b), 1 if out_int8 else 0, float(np.float32(s_y)), _ptr(z),
                                _ptr(y16), _ptr(y8))
    if rc == 5:
        raise OverflowError("W8A8 dot product exceeds the INT32 range")
    if rc != 0:
        raise ValueError("orc_gemv_w8a8_ex failed with code %d" % rc)
    return z, (y8 if out_int8 else y16.view(np.float16))


def linear_w8a8(M, N, K, X, ldx, s_x, W, ldw, s_W, bias=None, out_int8=False, s_y=1.0):
    """Batch of M tokens: (z int64 [M, N], Y [M, N]) with Y FP16 or int8 (out_int8);
    X is M x ldx int8, s_x [M] per-token scales."""
    X = np.ascontiguousarray(X, dtype=np.int8)
    W = np.ascontiguousarray(W, dtype=np.int8)
    s_x = np.ascontiguousarray(s_x, dtype=np.float32)
    s_W = np.ascontiguousarray(s_W, dtype=np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    z = np.zeros((M, N), dtype=np.int64)
    y16 = np.zeros((M, N), dtype=np.uint16)
    y8 = np.zeros((M, N), dtype=np.int8)
    rc = lib().orc_linear_w8a8(M, N, K, _ptr(X), ldx, _ptr(s_x), _ptr(W), ldw, _ptr(s_W), _ptr(b),
                               1 if out_int8 else 0, float(np.float32(s_y)), _ptr(z), _ptr(y16),
                               _ptr(y8), N)
    if rc == 5:
        raise OverflowError("W8A8 dot product exceeds the INT32 range")
    if rc != 0:
        raise ValueError("orc_linear_w8a8 failed with code %d" % rc)
    return z, (y8 if out_int8 else y16.view(np.float16))


def linear_w8a16(M, N, K, X_bits, ldx, W, ldw, s_W, bias=None):
    """Weight-only layer: (y float64 [M, N], absab [M, N]); X_bits are BF16 codes
    (uint16, M x ldx), W int8 N x ldw, s_W float32 [N]."""
    X = np.ascontiguousarray(X_bits, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.int8)
    s_W = np.ascontiguousarray(s_W, dtype=np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    y = np.zeros((M, N), dtype=np.float64)
    ab = np.zeros((M, N), dtype=np.float64)
    rc = lib().orc_linear_w8a16(M, N, K, _ptr(X), ldx, _ptr(W), ldw, _ptr(s_W), _ptr(b), _ptr(y), _ptr(ab))
    if rc != 0:
        raise ValueError("orc_linear_w8a16 failed with code %d" % rc)
    return y, ab


def threads_used() -> int:
    """Threads OpenMP will use (OMP_NUM_THREADS, else the usable cores)."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env:
        return int(env)
    return len(os.sched_getaffinity(0))
