"""linear_layer_gb300: GB300 (sm_103a) linear-layer hot path behind a C ABI.

This module is a thin ctypes binding over ``lib/liblinear_layer_gb300.so``: it
turns torch tensors (or raw integer device pointers) into pointers and calls the
C entry points declared in ``include/ll.h``.  Every step of the computation runs
in the library's CUDA kernels; there is no Python or CPU fallback.  If the
library has not been built, importing this package raises ImportError.

Python name          C entry point
------------------   -------------------------
gemm_f16             ll_gemm_f16
gemm_bf16            ll_gemm_bf16
gemm_fp8_blockscaled ll_gemm_fp8_blockscaled
gemm_f8_blockscaled_mixed ll_gemm_f8_blockscaled_mixed
gemm_mxf8            ll_gemm_mxf8
gemm_mxf8_workspace_size ll_gemm_mxf8_workspace_size
gemm_nvf4            ll_gemm_nvf4
gemm_nvf4_workspace_size ll_gemm_nvf4_workspace_size
linear_w8a8_gemv     ll_linear_w8a8_gemv
linear_w8a8_gemv_ex  ll_linear_w8a8_gemv_ex
linear_w8a8          ll_linear_w8a8
linear_w8a16         ll_linear_w8a16
linear_f16_w8a8_gemv ll_linear_f16_w8a8_gemv
quantize_per_token_f16 ll_quantize_per_token_f16
gemm_f16_noalloc     ll_gemm_f16_noalloc
gemm_workspace_size  ll_gemm_workspace_size
get_device_status    ll_get_device_status
set_wait_timeout_ns  ll_set_wait_timeout_ns
debug_timeout_probe  ll_debug_timeout_probe
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "liblinear_layer_gb300.so")

LL_OK, LL_ERR_INVALID_ARG, LL_ERR_MISALIGNED, LL_ERR_UNSUPPORTED = 0, 1, 2, 3
LL_ERR_WORKSPACE, LL_ERR_CUDA, LL_ERR_DEVICE_TIMEOUT, LL_ERR_NO_DEVICE = 4, 5, 6, 7
IN_F16, IN_BF16, IN_E4M3, IN_E5M2 = 0, 1, 2, 3
GEMV_OUT_F16, GEMV_OUT_I8 = 0, 1
OUT_F32, OUT_BF16, OUT_F16 = 0, 1, 2

# every symbol the header declares
EXPORTS = ["ll_gemm_workspace_size", "ll_gemm_f16", "ll_gemm_bf16", "ll_gemm_fp8_blockscaled",
           "ll_gemm_f16_noalloc", "ll_gemm_f8_blockscaled_mixed", "ll_gemm_mxf8",
           "ll_gemm_mxf8_workspace_size", "ll_gemm_nvf4", "ll_gemm_nvf4_workspace_size",
           "ll_linear_w8a8_gemv", "ll_linear_w8a8_gemv_ex", "ll_linear_f16_w8a8_gemv",
           "ll_linear_w8a8", "ll_linear_w8a16",
           "ll_quantize_per_token_f16", "ll_get_device_status", "ll_set_wait_timeout_ns",
           "ll_debug_timeout_probe", "ll_status_string", "ll_version"]


class LLError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s" % (where, status_string(status)))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("linear_layer_gb300: the CUDA library is not built (%s missing); "
                          "run `python -m linear_layer_gb300.build`" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    L.ll_gemm_workspace_size.restype = ctypes.c_size_t
    L.ll_gemm_workspace_size.argtypes = [i32, i32, i32, i64, i64, i32]
    dense = [i32, i32, i32, f32, vp, i64, vp, i64, f32, vp, i64, vp, i64, i32, vp, ctypes.c_size_t, vp]
    for name in ("ll_gemm_f16", "ll_gemm_bf16"):
        getattr(L, name).restype = i32
        getattr(L, name).argtypes = dense
    L.ll_gemm_f16_noalloc.restype = i32
    L.ll_gemm_f16_noalloc.argtypes = dense[:14] + [vp]
    L.ll_gemm_fp8_blockscaled.restype = i32
    L.ll_gemm_fp8_blockscaled.argtypes = [i32, i32, i32, f32, vp, i64, vp, i64, vp, i64, vp, i64,
                                          f32, vp, i64, vp, i64, i32, vp, ctypes.c_size_t, vp]
    L.ll_gemm_f8_blockscaled_mixed.restype = i32
    L.ll_gemm_f8_blockscaled_mixed.argtypes = [i32, i32] + L.ll_gemm_fp8_blockscaled.argtypes
    L.ll_gemm_mxf8_workspace_size.restype = ctypes.c_size_t
    L.ll_gemm_mxf8_workspace_size.argtypes = [i32, i32, i32, i64, i64]
    L.ll_gemm_mxf8.restype = i32
    L.ll_gemm_mxf8.argtypes = [i32, i32] + L.ll_gemm_fp8_blockscaled.argtypes
    L.ll_gemm_nvf4_workspace_size.restype = ctypes.c_size_t
    L.ll_gemm_nvf4_workspace_size.argtypes = [i32, i32, i32, i64, i64]
    L.ll_gemm_nvf4.restype = i32
    L.ll_gemm_nvf4.argtypes = L.ll_gemm_fp8_blockscaled.argtypes
    L.ll_linear_w8a8_gemv.restype = i32
    L.ll_linear_w8a8_gemv.argtypes = [i32, i32, vp, vp, vp, i64, vp, vp, vp, vp]
    L.ll_linear_w8a8_gemv_ex.restype = i32
    L.ll_linear_w8a8_gemv_ex.argtypes = [i32, i32, vp, vp, vp, i64, vp, vp, i32, vp, vp, vp, vp]
    L.ll_linear_w8a8.restype = i32
    L.ll_linear_w8a8.argtypes = [i32, i32, i32, vp, i64, vp, vp, i64, vp, vp, i32, vp, vp, i64, vp,
                                 i64, vp]
    L.ll_linear_w8a16.restype = i32
    L.ll_linear_w8a16.argtypes = [i32, i32, i32, vp, i64, vp, i64, vp, vp, i32, vp, i64, vp]
    L.ll_linear_f16_w8a8_gemv.restype = i32
    L.ll_linear_f16_w8a8_gemv.argtypes = [i32, i32, vp, vp, vp, vp, i64, vp, vp, i32, vp, vp, vp, vp]
    L.ll_quantize_per_token_f16.restype = i32
    L.ll_quantize_per_token_f16.argtypes = [i32, i32, vp, i64, vp, i64, vp, vp]
    L.ll_get_device_status.restype = i32
    L.ll_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    L.ll_set_wait_timeout_ns.restype = i32
    L.ll_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    L.ll_debug_timeout_probe.restype = i32
    L.ll_debug_timeout_probe.argtypes = [vp]
    L.ll_status_string.restype = ctypes.c_char_p
    L.ll_status_string.argtypes = [i32]
    L.ll_version.restype = ctypes.c_char_p
    L.ll_version.argtypes = []
    return L


lib = _load()


def status_string(status):
    return lib.ll_status_string(int(status)).decode()


def version():
    return lib.ll_version().decode()


def _p(x):
    """Device pointer of a CUDA torch tensor, an int (taken as a device address), or None.
    A tensor in host memory, or on another GPU than the current one (where every call
    runs), is refused: the library would use its address as memory of the current GPU."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("linear_layer_gb300: expected a CUDA tensor, got one on %s" % (x.device,))
    import torch
    if x.get_device() != torch.cuda.current_device():
        raise ValueError("linear_layer_gb300: tensor on %s, but the calls run on the current device cuda:%d"
                         % (x.device, torch.cuda.current_device()))
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status, where):
    if status != LL_OK:
        raise LLError(status, where)
    return status


def gemm_workspace_size(M, N, K, lda, ldb, in_type):
    return lib.ll_gemm_workspace_size(M, N, K, lda, ldb, in_type)


def _ws(workspace):
    if workspace is None:
        return None, 0
    if isinstance(workspace, tuple):
        return workspace
    return _p(workspace), workspace.numel() * workspace.element_size()


def gemm_f16(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd, d_type, workspace=None,
             stream=None):
    w, wb = _ws(workspace)
    return _check(lib.ll_gemm_f16(M, N, K, alpha, _p(A), lda, _p(B), ldb, beta, _p(C), ldc, _p(D),
                                  ldd, d_type, w, wb, _stream(stream)), "ll_gemm_f16")


def gemm_bf16(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd, d_type, workspace=None,
              stream=None):
    w, wb = _ws(workspace)
    return _check(lib.ll_gemm_bf16(M, N, K, alpha, _p(A), lda, _p(B), ldb, beta, _p(C), ldc, _p(D),
                                   ldd, d_type, w, wb, _stream(stream)), "ll_gemm_bf16")


def gemm_f16_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, D, ldd, d_type, stream=None):
    """ll_gemm_f16 without workspace: unaligned operands are repacked into the library's
    fixed 16 MiB device scratch (for callers that cannot allocate; calls must not
    overlap on the GPU)."""
    return _check(lib.ll_gemm_f16_noalloc(M, N, K, alpha, _p(A), lda, _p(B), ldb, beta, _p(C), ldc,
                                          _p(D), ldd, d_type, _stream(stream)),
                  "ll_gemm_f16_noalloc")


def gemm_fp8_blockscaled(M, N, K, alpha, A, lda, scale_a, ld_sa, B, ldb, scale_b, ld_sb, beta, C,
                         ldc, D, ldd, d_type, workspace=None, stream=None):
    w, wb = _ws(workspace)
    return _check(lib.ll_gemm_fp8_blockscaled(M, N, K, alpha, _p(A), lda, _p(scale_a), ld_sa, _p(B),
                                              ldb, _p(scale_b), ld_sb, beta, _p(C), ldc, _p(D), ldd,
                                              d_type, w, wb, _stream(stream)),
                  "ll_gemm_fp8_blockscaled")


def gemm_f8_blockscaled_mixed(a_type, b_type, M, N, K, alpha, A, lda, scale_a, ld_sa, B, ldb,
                              scale_b, ld_sb, beta, C, ldc, D, ldd, d_type, workspace=None,
                              stream=None):
    w, wb = _ws(workspace)
    return _check(lib.ll_gemm_f8_blockscaled_mixed(a_type, b_type, M, N, K, alpha, _p(A), lda,
                                                   _p(scale_a), ld_sa, _p(B), ldb, _p(scale_b),
                                                   ld_sb, beta, _p(C), ldc, _p(D), ldd, d_type, w,
                                                   wb, _stream(stream)),
                  "ll_gemm_f8_blockscaled_mixed")


def gemm_mxf8_workspace_size(M, N, K, lda, ldb):
    return lib.ll_gemm_mxf8_workspace_size(M, N, K, lda, ldb)


def gemm_mxf8(a_type, b_type, M, N, K, alpha, A, lda, scale_a, ld_sa, B, ldb, scale_b, ld_sb, beta, C, ldc,
              D, ldd, d_type, workspace=None, stream=None):
    """MX block-scaled 8-bit GEMM: scale_a (M x ld_sa) and scale_b (N x ld_sb) hold E8M0
    codes, one per 32-wide K block of a row of A / a column of B."""
    w, wb = _ws(workspace)
    return _check(lib.ll_gemm_mxf8(a_type, b_type, M, N, K, alpha, _p(A), lda, _p(scale_a), ld_sa, _p(B), ldb,
                                   _p(scale_b), ld_sb, beta, _p(C), ldc, _p(D), ldd, d_type, w, wb,
                                   _stream(stream)), "ll_gemm_mxf8")


def gemm_nvf4_workspace_size(M, N, K, lda, ldbt):
    return lib.ll_gemm_nvf4_workspace_size(M, N, K, lda, ldbt)


def gemm_nvf4(M, N, K, alpha, A, lda, scale_a, ld_sa, Bt, ldbt, scale_b, ld_sb, beta, C, ldc, D, ldd, d_type,
              workspace=None, stream=None):
    """NVFP4 GEMM: A (M x K) and Bt (N x K, B transposed) hold E2M1 codes two per byte,
    pitches in elements; scale_a / scale_b hold UE4M3 codes, one per 16-wide K block."""
    w, wb = _ws(workspace)
    return _check(lib.ll_gemm_nvf4(M, N, K, alpha, _p(A), lda, _p(scale_a), ld_sa, _p(Bt), ldbt, _p(scale_b),
                                   ld_sb, beta, _p(C), ldc, _p(D), ldd, d_type, w, wb, _stream(stream)),
                  "ll_gemm_nvf4")


def linear_w8a8_gemv(N, K, x, x_scale, W, ldw, w_scale, y, z_out=None, stream=None):
    return _check(lib.ll_linear_w8a8_gemv(N, K, _p(x), _p(x_scale), _p(W), ldw, _p(w_scale), _p(y),
                                          _p(z_out), _stream(stream)), "ll_linear_w8a8_gemv")


def linear_w8a8_gemv_ex(N, K, x, x_scale, W, ldw, w_scale, bias, y_type, y_scale, y, z_out=None,
                        stream=None):
    return _check(lib.ll_linear_w8a8_gemv_ex(N, K, _p(x), _p(x_scale), _p(W), ldw, _p(w_scale),
                                             _p(bias), y_type, _p(y_scale), _p(y), _p(z_out),
                                             _stream(stream)), "ll_linear_w8a8_gemv_ex")


def linear_w8a8(M, N, K, X, ldx, x_scale, W, ldw, w_scale, bias, y_type, y_scale, Y, ldy,
                z_out=None, ldz=0, stream=None):
    return _check(lib.ll_linear_w8a8(M, N, K, _p(X), ldx, _p(x_scale), _p(W), ldw, _p(w_scale),
                                     _p(bias), y_type, _p(y_scale), _p(Y), ldy, _p(z_out), ldz,
                                     _stream(stream)), "ll_linear_w8a8")


def linear_w8a16(M, N, K, X, ldx, W, ldw, w_scale, bias, y_type, Y, ldy, stream=None):
    return _check(lib.ll_linear_w8a16(M, N, K, _p(X), ldx, _p(W), ldw, _p(w_scale), _p(bias), y_type,
                                      _p(Y), ldy, _stream(stream)), "ll_linear_w8a16")


def linear_f16_w8a8_gemv(N, K, x, x_q, x_scale, W, ldw, w_scale, bias, y_type, y_scale, y,
                         z_out=None, stream=None):
    return _check(lib.ll_linear_f16_w8a8_gemv(N, K, _p(x), _p(x_q), _p(x_scale), _p(W), ldw,
                                              _p(w_scale), _p(bias), y_type, _p(y_scale), _p(y),
                                              _p(z_out), _stream(stream)), "ll_linear_f16_w8a8_gemv")


def quantize_per_token_f16(M, K, x, ldx, q, ldq, scale, stream=None):
    return _check(lib.ll_quantize_per_token_f16(M, K, _p(x), ldx, _p(q), ldq, _p(scale),
                                                _stream(stream)), "ll_quantize_per_token_f16")


def get_device_status(stream=None):
    """(status, raw word): synchronises the stream, reads and clears the status word."""
    word = ctypes.c_uint32(0)
    st = lib.ll_get_device_status(_stream(stream), ctypes.byref(word))
    return st, word.value


def set_wait_timeout_ns(ns):
    return _check(lib.ll_set_wait_timeout_ns(int(ns)), "ll_set_wait_timeout_ns")


def debug_timeout_probe(stream=None):
    return _check(lib.ll_debug_timeout_probe(_stream(stream)), "ll_debug_timeout_probe")
