"""ll_gemm_f16_noalloc, the FP16 GEMM for callers that cannot allocate device memory
(runtimes whose allocator owns all device memory, plugin interfaces that pass
neither an allocator nor a workspace, latency-critical paths where allocating is not
allowed), checked against ll_gemm_f16 with a caller-provided workspace.

The new entry point repacks operands whose row pitch is not a multiple of 16 bytes
into a fixed 16 MiB scratch array inside the library instead of the caller's
workspace, with the same layout and the same kernels, so its output must equal the
existing entry point's bit for bit (these shapes are too small for the stream-K split of
the last wave, the one schedule that needs more workspace than the repacks and that
this entry point never uses).  Two calls run in a row, with different shapes and
inputs; the second call's repacked A lies over the bytes where the first call's
repacked B was, so a repack that left any earlier bytes in place would change its
output.  This file is collected last so that a run stopping at its first failure has
already run every other test; it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


def _one_call(M, N, K, lda, ldb, out, seed, alpha, beta):
    import linear_layer_gb300 as ll
    dev = torch.device("cuda:0")
    A = wl.f16_uniform(M, K, seed, ld=lda)
    B = wl.f16_uniform(K, N, seed + 1, ld=ldb)
    C = wl.f32_normal(M, N, seed + 2)
    tA = torch.from_numpy(A.view(np.int16)).to(dev)
    tB = torch.from_numpy(B.view(np.int16)).to(dev)
    tC = torch.from_numpy(C).to(dev)
    dt, code = {"f32": (torch.float32, ll.OUT_F32), "bf16": (torch.bfloat16, ll.OUT_BF16)}[out]
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
    assert not torch.isnan(D_old.float()).any()
    # same repack layout, same kernels: the outputs are bit-identical
    assert torch.equal(D_new.view(torch.int32 if out == "f32" else torch.int16),
                       D_old.view(torch.int32 if out == "f32" else torch.int16))


def test_noalloc_matches_workspace_entry_two_calls_in_a_row():
    # 1st call: A pitch 402 bytes and B pitch 666 bytes both need the repack; in the
    # scratch, A takes bytes [0, 120064) and B starts at byte 120064
    _one_call(300, 333, 200, lda=201, ldb=333, out="f32", seed=41, alpha=0.5, beta=-1.25)
    # 2nd call: another shape and inputs; its repacked A (517 x 136 FP16, 140624 bytes)
    # covers the start of the first call's B region, and B is repacked after it
    _one_call(517, 1003, 136, lda=137, ldb=1003, out="bf16", seed=51, alpha=1.0, beta=1.0)


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
