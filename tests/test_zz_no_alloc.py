"""ll_gemm_f16_noalloc, the FP16 GEMM for callers that cannot allocate device memory
(runtimes whose allocator owns all device memory, plugin interfaces that pass
neither an allocator nor a workspace, latency-critical paths where allocating is not
allowed), checked against ll_gemm_f16 with a caller-provided workspace.

The new entry point repacks operands whose row pitch is not a multiple of 16 bytes
into a fixed 16 MiB scratch array inside the library instead of the caller's
workspace.  Two calls in a row, with different shapes and inputs, must each match the
existing entry point within the tolerance the other GEMM tests use; the second call
also shows that what the first call left in the shared scratch does not leak into it.
This file is collected last so that a run stopping at its first failure has already
run every other test; it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


def _bound_check(D_new, D_old, A, B, K, u_out, lda, ldb, M, N):
    """|D_new - D_old| within the GEMM tolerance scale 1e-2 sqrt(K/256) (|A||B|) + 1e-6."""
    Ad = torch.from_numpy(A.view(np.float16)[:, :K].astype(np.float32))
    Bd = torch.from_numpy(B.view(np.float16)[:, :N].astype(np.float32))
    absab = (Ad.abs().double() @ Bd.abs().double()).numpy()
    new = D_new.float().cpu().numpy().astype(np.float64)[:, :N]
    old = D_old.float().cpu().numpy().astype(np.float64)[:, :N]
    bound = 1e-2 * np.sqrt(K / 256.0) * absab + 1e-6 + u_out * np.abs(old)
    assert np.all(np.abs(new - old) <= bound)
    nold = np.linalg.norm(old)
    assert np.linalg.norm(new - old) <= (1e-3 + u_out * (1 + 1e-3)) * nold


def _one_call(M, N, K, lda, ldb, out, seed, alpha, beta):
    import linear_layer_gb300 as ll
    dev = torch.device("cuda:0")
    A = wl.f16_uniform(M, K, seed, ld=lda)
    B = wl.f16_uniform(K, N, seed + 1, ld=ldb)
    C = wl.f32_normal(M, N, seed + 2)
    tA = torch.from_numpy(A.view(np.int16)).to(dev)
    tB = torch.from_numpy(B.view(np.int16)).to(dev)
    tC = torch.from_numpy(C).to(dev)
    dt, code, u_out = {"f32": (torch.float32, ll.OUT_F32, 0.0),
                       "bf16": (torch.bfloat16, ll.OUT_BF16, 2.0 ** -8)}[out]
    D_old = torch.full((M, N), float("nan"), dtype=dt, device=dev)
    D_new = torch.full((M, N), float("nan"), dtype=dt, device=dev)
    need = ll.gemm_workspace_size(M, N, K, lda, ldb, ll.IN_F16)
    assert need > 0  # these shapes do need a repack
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    # the existing entry point, with the caller's workspace
    st = ll.lib.ll_gemm_f16(M, N, K, alpha, tA.data_ptr(), lda, tB.data_ptr(), ldb, beta,
                            tC.data_ptr(), N, D_old.data_ptr(), N, code, ws.data_ptr(),
                            ctypes.c_size_t(need), stream)
    assert st == ll.LL_OK
    # the allocation-free entry point, through the C ABI
    st = ll.lib.ll_gemm_f16_noalloc(M, N, K, alpha, tA.data_ptr(), lda, tB.data_ptr(), ldb, beta,
                                    tC.data_ptr(), N, D_new.data_ptr(), N, code, stream)
    assert st == ll.LL_OK, ll.status_string(st)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, word
    assert not torch.isnan(D_new.float()).any()
    _bound_check(D_new, D_old, A, B, K, u_out, lda, ldb, M, N)


def test_noalloc_matches_workspace_entry_two_calls_in_a_row():
    # 1st call: B pitch 666 bytes and A pitch 402 bytes both need the repack
    _one_call(300, 333, 200, lda=201, ldb=333, out="f32", seed=41, alpha=0.5, beta=-1.25)
    # 2nd call: another shape and inputs over the same scratch (only B repacked)
    _one_call(517, 1003, 136, lda=136, ldb=1003, out="bf16", seed=51, alpha=1.0, beta=1.0)


def test_noalloc_rejects_requests_beyond_the_scratch():
    import linear_layer_gb300 as ll
    dev = torch.device("cuda:0")
    M, N, K = 64, 4099, 4096  # B repack: 4096 * 4104 * 2 bytes > 16 MiB
    t = torch.zeros(K * N + 64, dtype=torch.float16, device=dev)
    D = torch.zeros((M, N), dtype=torch.float32, device=dev)
    st = ll.lib.ll_gemm_f16_noalloc(M, N, K, 1.0, t.data_ptr(), K, t.data_ptr(), N, 0.0, None, N,
                                    D.data_ptr(), N, ll.OUT_F32,
                                    torch.cuda.current_stream().cuda_stream)
    assert st == ll.LL_ERR_WORKSPACE
