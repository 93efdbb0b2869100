"""Failure detection without a GPU fault: a bounded wait on a barrier phase that nothing
completes runs out, the kernel records LL_ERR_DEVICE_TIMEOUT in the device status word and
returns; the context stays usable and the next GEMM runs and reports LL_OK."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import check_close, up

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(orc):
    import linear_layer_gb300 as ll
    st, _ = ll.get_device_status()
    assert st == ll.LL_OK
    ll.set_wait_timeout_ns(50_000_000)  # 50 ms
    try:
        ll.debug_timeout_probe()
        st, word = ll.get_device_status()
    finally:
        ll.set_wait_timeout_ns(2_000_000_000)
    assert st == ll.LL_ERR_DEVICE_TIMEOUT
    assert (word >> 8) & 0xFF == 4  # the probe's role
    st, word = ll.get_device_status()  # cleared by the read
    assert st == ll.LL_OK and word == 0
    M, N, K = 128, 256, 64
    A, B, _ = wl.gemm_inputs("f16", M, N, K, 0.0)
    D = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ll.gemm_f16(M, N, K, 1.0, up(A), K, up(B), N, 0.0, None, N, D, N, ll.OUT_F32)
    st, _ = ll.get_device_status()
    assert st == ll.LL_OK
    ref, absab = orc.gemm("f16", M, N, K, 1.0, A.ravel(), K, B.ravel(), N)
    check_close(D.cpu().numpy(), ref, absab, K, "f32", "f16", "after timeout")


def test_invalid_timeout_rejected():
    import linear_layer_gb300 as ll
    with pytest.raises(ll.LLError):
        ll.set_wait_timeout_ns(0)
