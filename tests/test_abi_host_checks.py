"""Host-side argument checks of the C ABI, run where the library can see no GPU.

Every entry point validates its arguments before it looks for a device, so each
invalid request must come back with its documented status code (and an empty
request with LL_OK) without a GPU.  The pointers here are fake addresses that no
kernel may ever see, so the checks run in a child process started with
CUDA_VISIBLE_DEVICES set to the empty string: the CUDA driver then shows that process
no device at all, whatever the machine has, and a request that a faulty check let
through can only come back as "no device".  The child first confirms that the
library reports no device, and runs nothing otherwise.  (The GPU suite checks the
same rejections with real tensors.)"""
import os
import subprocess
import sys
import traceback

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
P = 0x7F0000000000  # a 256-byte-aligned stand-in address, never dereferenced


def _load_library():
    import importlib.util
    spec = importlib.util.spec_from_file_location("_ll_build", os.path.join(ROOT, "linear_layer_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    sys.path.insert(0, ROOT)
    import linear_layer_gb300
    return linear_layer_gb300


CHECKS = []


def check(fn):
    CHECKS.append(fn.__name__)
    return fn


def _child_main():
    """Entry of the device-less child: run every check, report one line per check."""
    assert os.environ.get("CUDA_VISIBLE_DEVICES") == ""
    ll = _load_library()
    st, _ = ll.lib.ll_get_device_status(None, None), None
    if st not in (ll.LL_ERR_NO_DEVICE, ll.LL_ERR_CUDA):
        print("ABORT the library sees a device (status %d): no fake address is passed" % st)
        return 3
    mod = sys.modules[__name__]
    for name in CHECKS:
        try:
            getattr(mod, name)(ll)
            print("OK %s" % name)
        except Exception:
            print("FAIL %s %s" % (name, traceback.format_exc().replace("\n", " | ")))
    return 0


@pytest.fixture(scope="module")
def child_results():
    _load_library()  # build in this process, so the child only loads
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    code = ("import sys; sys.path.insert(0, %r); sys.path.insert(0, %r); "
            "import test_abi_host_checks as t; sys.exit(t._child_main())" % (ROOT, os.path.join(ROOT, "tests")))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    out = r.stdout
    assert r.returncode == 0, "child exited %d: %s %s" % (r.returncode, out[-2000:], r.stderr[-2000:])
    res = {}
    for line in out.splitlines():
        parts = line.split(" ", 2)
        if parts[0] in ("OK", "FAIL") and len(parts) >= 2:
            res[parts[1]] = line
    return res


def _gemm(ll, M=64, N=64, K=64, A=P, lda=64, B=P, ldb=64, beta=0.0, C=None, ldc=64, D=P + 0x100000,
          ldd=64, d_type=0, fn="ll_gemm_f16", ws=None, ws_bytes=0):
    return getattr(ll.lib, fn)(M, N, K, 1.0, A, lda, B, ldb, beta, C, ldc, D, ldd, d_type, ws, ws_bytes, None)


def _no_device(ll, st):
    return st in (ll.LL_ERR_NO_DEVICE, ll.LL_ERR_CUDA)


@check
def check_gemm_rejections(ll):
    E, MIS = ll.LL_ERR_INVALID_ARG, ll.LL_ERR_MISALIGNED
    assert _gemm(ll, M=-1) == E
    assert _gemm(ll, K=-1) == E
    assert _gemm(ll, d_type=7) == E
    assert _gemm(ll, D=None) == E
    assert _gemm(ll, ldd=63) == E
    assert _gemm(ll, beta=1.0, C=None) == E                               # C needed when beta != 0
    assert _gemm(ll, beta=1.0, C=P + 0x100000, d_type=ll.OUT_BF16) == E   # in place only for FP32
    assert _gemm(ll, beta=1.0, C=P + 0x100000, ldc=64, ldd=65, d_type=ll.OUT_F32) == E
    assert _gemm(ll, lda=63) == E
    assert _gemm(ll, A=None) == E
    assert _gemm(ll, D=P + 0x100002, d_type=ll.OUT_F32) == MIS            # D not on a 4-byte boundary
    assert _gemm(ll, D=P + 0x100001, d_type=ll.OUT_BF16) == MIS           # nor a 2-byte one
    assert _gemm(ll, beta=0.5, C=P + 0x200002) == MIS                     # C read: 4-byte aligned
    assert _gemm(ll, fn="ll_gemm_bf16", ldb=10) == E


@check
def check_gemm_workspace_may_not_overlap(ll):
    """A 16-bit GEMM may write its workspace (stream-K partial tiles) even when nothing is
    repacked, so a workspace that shares bytes with D or an input is rejected."""
    E = ll.LL_ERR_INVALID_ARG
    D = P + 0x100000
    assert _gemm(ll, ws=D + 0x800, ws_bytes=1 << 20) == E                    # inside D
    assert _gemm(ll, ws=P + 0x40, ws_bytes=1 << 20, fn="ll_gemm_bf16") == E  # inside A and B
    assert _no_device(ll, _gemm(ll, ws=P + 0x400000, ws_bytes=1 << 20))     # disjoint: accepted


@check
def check_gemm_empty_requests_need_no_device(ll):
    assert _gemm(ll, M=0) == ll.LL_OK
    assert _gemm(ll, N=0, D=None) == ll.LL_OK
    assert _gemm(ll, M=0, fn="ll_gemm_bf16") == ll.LL_OK


@check
def check_gemm_valid_request_reports_the_missing_device(ll):
    assert _no_device(ll, _gemm(ll))
    assert _no_device(ll, _gemm(ll, lda=65))  # a repack is needed, but the device check comes first


def _fp8(ll, sA=P + 0x300000, ld_sa=1, sB=P + 0x400000, ld_sb=1, K=128, N=128):
    return ll.lib.ll_gemm_fp8_blockscaled(64, N, K, 1.0, P, K, sA, ld_sa, P, N, sB, ld_sb, 0.0, None, N,
                                          P + 0x100000, N, ll.OUT_BF16, None, 0, None)


@check
def check_fp8_scale_checks(ll):
    E, MIS = ll.LL_ERR_INVALID_ARG, ll.LL_ERR_MISALIGNED
    assert _fp8(ll, sA=None) == E
    assert _fp8(ll, sB=None) == E
    assert _fp8(ll, K=129, ld_sa=1) == E   # ceil(129 / 128) = 2 K blocks per row of scale_a
    assert _fp8(ll, N=129, ld_sb=1) == E   # and 2 column blocks per row of scale_b
    assert _fp8(ll, sA=P + 0x300002) == MIS
    assert _no_device(ll, _fp8(ll))


@check
def check_gemv_checks(ll):
    E = ll.LL_ERR_INVALID_ARG
    g = ll.lib.ll_linear_w8a8_gemv
    assert g(-1, 64, P, P, P, 64, P, P, None, None) == E
    assert g(16, 131072, P, P, P, 131072, P, P, None, None) == E   # int32 sums could overflow
    assert g(16, 64, P, None, P, 64, P, P, None, None) == E        # x_scale
    assert g(16, 64, P, P, P, 63, P, P, None, None) == E           # ldw < K
    assert g(16, 64, None, P, P, 64, P, P, None, None) == E        # x with K > 0
    assert g(0, 64, None, None, None, 0, None, None, None, None) == ll.LL_OK
    assert _no_device(ll, g(16, 64, P, P, P, 64, P, P + 0x100000, None, None))
    ex = ll.lib.ll_linear_w8a8_gemv_ex
    assert ex(16, 64, P, P, P, 64, P, None, 5, None, P, None, None) == E              # output type
    assert ex(16, 64, P, P, P, 64, P, None, ll.GEMV_OUT_I8, None, P, None, None) == E  # INT8 needs s_y


@check
def check_token_layer_checks(ll):
    E = ll.LL_ERR_INVALID_ARG
    f = ll.lib.ll_linear_w8a8
    args = dict(M=4, N=16, K=64, X=P, ldx=64, xs=P, W=P, ldw=64, ws=P, bias=None, yt=ll.GEMV_OUT_F16, ys=None,
                Y=P + 0x100000, ldy=16, Z=None, ldz=16)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["M"], a["N"], a["K"], a["X"], a["ldx"], a["xs"], a["W"], a["ldw"], a["ws"], a["bias"], a["yt"],
                 a["ys"], a["Y"], a["ldy"], a["Z"], a["ldz"], None)
    assert call(M=-1) == E
    assert call(ldx=63) == E
    assert call(ldy=15) == E
    assert call(Z=P + 0x200000, ldz=15) == E
    assert call(yt=ll.GEMV_OUT_I8) == E
    assert call(M=0) == ll.LL_OK
    assert _no_device(ll, call())
    w = ll.lib.ll_linear_w8a16
    assert w(2, 16, 64, P, 64, P, 64, P, None, 9, P, 16, None) == E        # output type
    assert w(2, 16, 64, P, 63, P, 64, P, None, ll.OUT_BF16, P, 16, None) == E   # ldx < K
    assert w(0, 16, 64, P, 64, P, 64, P, None, ll.OUT_BF16, P, 16, None) == ll.LL_OK


@check
def check_noalloc_and_quantiser_checks(ll):
    E, MIS = ll.LL_ERR_INVALID_ARG, ll.LL_ERR_MISALIGNED
    n = ll.lib.ll_gemm_f16_noalloc

    def call(M=64, D=P + 0x100000, d_type=0, lda=64, beta=0.0, C=None):
        return n(M, 64, 64, 1.0, P, lda, P, 64, beta, C, 64, D, 64, d_type, None)
    assert call(M=-1) == E
    assert call(lda=10) == E
    assert call(D=P + 0x100002) == MIS
    assert call(M=0) == ll.LL_OK
    assert _no_device(ll, call())
    q = ll.lib.ll_quantize_per_token_f16
    assert q(-1, 64, P, 64, P, 64, P, None) == E
    assert q(4, 64, P, 63, P, 64, P, None) == E   # ldx < K
    assert _no_device(ll, q(4, 64, P, 64, P + 0x100000, 64, P + 0x200000, None))


@check
def check_gemm_output_overlap(ll):
    """D may share no byte with A, B, C (other than D == C in place), the FP8 scales or a
    workspace that a repack writes; extents with the same pitch are compared row by row."""
    E = ll.LL_ERR_INVALID_ARG
    Q = P + 0x100000
    assert _gemm(ll, D=P + 64) == E                      # inside A's first row
    assert _gemm(ll, D=P + 64 * 2 * 63) == E             # A's last row
    assert _gemm(ll, B=Q + 64 * 4 * 63, D=Q) == E        # B starts in D's last row
    assert _no_device(ll, _gemm(ll, D=P + 64 * 2 * 64))  # right after A (and B) end
    # C and D as column blocks of one FP32 matrix with pitch 128: disjoint, allowed
    assert _no_device(ll, _gemm(ll, beta=1.0, C=Q, ldc=128, D=Q + 256, ldd=128))
    # ... but shifted by 32 columns they share columns 32..63 of every row
    assert _gemm(ll, beta=1.0, C=Q, ldc=128, D=Q + 128, ldd=128) == E
    # D's rows in the padding of C's (pitch 128 floats, D 64 floats wide) with another pitch
    # are disjoint but not provably so for different pitches: rejected
    assert _gemm(ll, beta=1.0, C=Q, ldc=128, D=Q + 256, ldd=192) == E
    # in place D == C with the same pitch stays allowed
    assert _no_device(ll, _gemm(ll, beta=1.0, C=Q, ldc=64, D=Q, ldd=64))
    # a workspace that the repack would write may not cover an operand or D
    f = ll.lib.ll_gemm_f16
    assert f(64, 64, 64, 1.0, P, 65, P + 0x10000, 64, 0.0, None, 64, Q, 64, 0, P + 0x8000,
             0x10000, None) == E                         # overlaps B
    assert _no_device(ll, f(64, 64, 64, 1.0, P, 65, P + 0x10000, 64, 0.0, None, 64, Q, 64, 0,
                            P + 0x200000, 0x10000, None))
    # the FP8 scales are inputs too
    assert _fp8(ll, sA=P + 0x100000 + 4) == E


@check
def check_layer_output_overlap(ll):
    E = ll.LL_ERR_INVALID_ARG
    Y = P + 0x100000
    g = ll.lib.ll_linear_w8a8_gemv
    assert g(16, 64, P, P, P, 64, P, P, None, None) == E               # y over x
    assert g(16, 64, P, P + 0x800, P, 64, P + 0x900, Y, Y + 16, None) == E  # z over y
    assert _no_device(ll, g(16, 64, P, P + 0x800, P, 64, P + 0x900, Y, Y + 32, None))
    fused = ll.lib.ll_linear_f16_w8a8_gemv
    # x_q (an output) over x (an input)
    assert fused(16, 64, P, P + 64, P + 0x800, P + 0x1000, 64, P + 0x2000, None, 0, None, Y, None, None) == E
    assert _no_device(ll, fused(16, 64, P, P + 128, P + 0x800, P + 0x1000, 64, P + 0x2000, None, 0, None, Y,
                                None, None))
    f = ll.lib.ll_linear_w8a8
    # Y (M x N FP16, pitch 32 bytes) over X (M x K int8)
    assert f(4, 16, 64, P, 64, P + 0x800, P + 0x1000, 64, P + 0x2000, None, 0, None, P + 64, 16, None, 16,
             None) == E
    assert _no_device(ll, f(4, 16, 64, P, 64, P + 0x800, P + 0x1000, 64, P + 0x2000, None, 0, None, Y, 16,
                            None, 16, None))
    w = ll.lib.ll_linear_w8a16
    assert w(2, 16, 64, P, 64, P + 0x1000, 64, P + 0x2000, None, ll.OUT_BF16, P + 0x1000 + 64, 16, None) == E
    assert _no_device(ll, w(2, 16, 64, P, 64, P + 0x1000, 64, P + 0x2000, None, ll.OUT_BF16, Y, 16, None))
    q = ll.lib.ll_quantize_per_token_f16
    assert q(4, 64, P, 64, P + 0x100000, 64, P + 0x100000 + 8, None) == E   # scale over q


@check
def check_mx_gemm(ll):
    """ll_gemm_mxf8: element types, scale pointers and pitches, and the workspace it always
    needs for the rearranged scale codes."""
    E = ll.LL_ERR_INVALID_ARG
    f = ll.lib.ll_gemm_mxf8
    Q, SA, SB, WS = P + 0x100000, P + 0x200000, P + 0x300000, P + 0x400000
    need = ll.lib.ll_gemm_mxf8_workspace_size(64, 64, 100, 100, 64)
    assert need >= 64 * 4 * 512 // 64  # scale blocks of one 128-row block of A and 256 columns of B

    def call(at=2, bt=2, K=100, ld_sa=4, ld_sb=4, sa=SA, sb=SB, ws=WS, wsb=None, D=Q):
        return f(at, bt, 64, 64, K, 1.0, P, K, sa, ld_sa, P, 64, sb, ld_sb, 0.0, None, 64, D, 64, ll.OUT_BF16, ws,
                 need if wsb is None else wsb, None)
    assert call(at=0) == E                  # FP16 is not an MX element type here
    assert call(bt=7) == E
    assert call(sa=None) == E
    assert call(ld_sb=3) == E               # ceil(100 / 32) = 4 K blocks per row of scales
    # a missing or short workspace is reported after the device check (as for a repack)
    assert _no_device(ll, call(ws=None, wsb=0))
    assert _no_device(ll, call(wsb=need - 1))
    assert call(D=SA + 2) == E              # D over scale_a
    assert call(ws=P + 0x10) == E           # workspace over A
    assert _no_device(ll, call())
    assert _no_device(ll, call(K=0, ws=None, wsb=0))  # K == 0: D = beta * C, no workspace


@check
def check_nvf4_gemm(ll):
    """ll_gemm_nvf4: even K and pitches (rows start on bytes), pitches in elements, scale
    pitches of ceil(K/16), and the workspace for the rearranged scale codes."""
    E = ll.LL_ERR_INVALID_ARG
    f = ll.lib.ll_gemm_nvf4
    Q, SA, SB, WS = P + 0x100000, P + 0x200000, P + 0x300000, P + 0x400000
    need = ll.lib.ll_gemm_nvf4_workspace_size(64, 64, 96, 96, 96)
    # pitch 48 bytes: no repack; scale blocks of one 128-row block of A (16 codes per row)
    # and one 256-column block of B
    assert need == 128 * 16 + 256 * 16 + 512
    assert ll.lib.ll_gemm_nvf4_workspace_size(64, 64, 96, 100, 96) > need  # 50-byte rows of A

    def call(K=96, lda=96, ldbt=96, ld_sa=6, ld_sb=6, sa=SA, ws=WS, wsb=None, D=Q):
        return f(64, 64, K, 1.0, P, lda, sa, ld_sa, P + 0x80000, ldbt, SB, ld_sb, 0.0, None, 64, D, 64,
                 ll.OUT_F32, ws, need if wsb is None else wsb, None)
    assert call(K=95) == E                  # odd K: a row would end inside a byte
    assert call(lda=97) == E                # odd pitch
    assert call(ldbt=95) == E
    assert call(lda=94) == E                # pitch below K
    assert call(ld_sa=5) == E               # ceil(96 / 16) = 6 scale codes per row
    assert call(ld_sb=5) == E
    assert call(sa=None) == E
    assert call(D=SB + 4) == E              # D over scale_b
    assert call(ws=P + 0x10) == E           # workspace over A (64 rows x 48 bytes)
    assert _no_device(ll, call(ws=None, wsb=0))
    assert _no_device(ll, call())
    assert _no_device(ll, call(ws=P + 64 * 48))  # just past A


@pytest.mark.parametrize("name", CHECKS)
def test_host_check_in_device_less_child(child_results, name):
    line = child_results.get(name)
    assert line is not None, "check %s did not run" % name
    assert line.startswith("OK "), line
