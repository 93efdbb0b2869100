"""GPU parity of the CTA-pair 16-bit GEMM when its last partial wave of tiles is split by
K ranges across all CTA pairs (stream-K; used when the caller's workspace has room for the
partial tiles, ll_gemm_workspace_size counting them): every element against the oracle,
for tails in M, N and K, alpha / beta, every output type, pieces that cross tile
boundaries and tiles with several pieces; outputs bit-identical from run to run; and the
same problems without that workspace (the last wave as 256 x 128 halves) within the same
tolerance of the oracle."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import assert_fully_written, check_all_rows, out_code, out_tensor, up

pytestmark = pytest.mark.gpu


def _run(orc, kind, M, N, K, alpha, beta, out, with_ws=True, seed=0):
    import linear_layer_gb300 as ll
    A = wl.operand(kind, M, K, wl.SEED_A + seed)
    B = wl.operand(kind, K, N, wl.SEED_B + seed)
    C = wl.f32_normal(M, N, wl.SEED_C + seed) if beta != 0.0 else None
    tD = out_tensor(M, N, out)
    in_type = ll.IN_F16 if kind == "f16" else ll.IN_BF16
    need = ll.gemm_workspace_size(M, N, K, K, N, in_type)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda") if (need and with_ws) else None
    fn = ll.gemm_f16 if kind == "f16" else ll.gemm_bf16
    fn(M, N, K, alpha, up(A), K, up(B), N, beta, up(C), N, tD, N, out_code(out), workspace=ws)
    st, word = ll.get_device_status()
    assert st == ll.LL_OK, "device status %s (word %#x)" % (ll.status_string(st), word)
    what = "%s %dx%dx%d%s" % (kind, M, N, K, "" if with_ws else " (no stream-K)")
    assert_fully_written(tD, M, N, what)
    Cf = None if C is None else C.ravel()
    check_all_rows(tD.float().cpu().numpy(),
                   lambda r: orc.gemm(kind, M, N, K, alpha, A.ravel(), K, B.ravel(), N, beta, Cf, N, rows=r),
                   M, N, K, out, kind, what)
    return tD, need


# shapes whose schedule on 76 CTA pairs leaves a last partial wave of at least 19 tiles:
# 256 tiles (28 left, 64 K blocks), 144 (68 left, 8 K blocks: about one piece per tile),
# 256 with tails in M, N and K (16 K blocks), 180 with N and K tails (13 K blocks)
@pytest.mark.parametrize("kind,M,N,K,alpha,beta,out", [
    ("bf16", 4096, 4096, 4096, 1.0, 1.0, "bf16"),
    ("f16", 3072, 3072, 512, 0.5, -1.25, "f32"),
    ("bf16", 4000, 4000, 1000, 1.0, 0.0, "f16"),
    ("f16", 2304, 5120, 776, 1.5, 0.75, "f32")])
def test_streamk_tail(orc, kind, M, N, K, alpha, beta, out):
    _, need = _run(orc, kind, M, N, K, alpha, beta, out)
    assert need > 0  # the workspace size counts the partial tiles


def test_streamk_deterministic(orc):
    a, _ = _run(orc, "bf16", 4096, 4096, 4096, 1.0, 1.0, "f32", seed=3)
    b, _ = _run(orc, "bf16", 4096, 4096, 4096, 1.0, 1.0, "f32", seed=3)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_without_streamk_workspace(orc):
    # no workspace: the same problem with the last wave as halves, also within tolerance
    _run(orc, "bf16", 4096, 4096, 4096, 1.0, 1.0, "bf16", with_ws=False)


def test_one_byte_less_turns_the_split_off():
    """The split runs exactly when the workspace reaches the size ll_gemm_workspace_size
    reports: with one byte less the call schedules the last wave as halves, so its output
    equals the no-workspace call's bit for bit."""
    import linear_layer_gb300 as ll
    M = N = K = 4096
    A = up(wl.operand("bf16", M, K, 91))
    B = up(wl.operand("bf16", K, N, 92))
    C = up(wl.f32_normal(M, N, 93))
    need = ll.gemm_workspace_size(M, N, K, K, N, ll.IN_BF16)
    assert need > 0
    outs = []
    for ws in (None, torch.empty(need - 1, dtype=torch.uint8, device="cuda")):
        tD = out_tensor(M, N, "f32")
        ll.gemm_bf16(M, N, K, 1.0, A, K, B, N, 1.0, C, N, tD, N, ll.OUT_F32, workspace=ws)
        st, word = ll.get_device_status()
        assert st == ll.LL_OK, "device status %s (word %#x)" % (ll.status_string(st), word)
        outs.append(tD)
    assert torch.equal(outs[0].view(torch.int32), outs[1].view(torch.int32))
