"""The C-ABI library loads on a machine without a GPU and exports every entry point
include/ll.h declares (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "ll.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ll_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def built_lib():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_ll_build", os.path.join(ROOT, "linear_layer_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build()


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ["ll_gemm_f16", "ll_gemm_bf16", "ll_gemm_fp8_blockscaled", "ll_linear_w8a8_gemv",
              "ll_gemm_workspace_size", "ll_get_device_status"]:
        assert n in names


def test_library_exports_every_declared_symbol(built_lib):
    lib = ctypes.CDLL(built_lib)
    for name in _declared():
        assert hasattr(lib, name), name


def test_python_binding_matches_header(built_lib):
    import linear_layer_gb300 as ll
    assert sorted(ll.EXPORTS) == _declared()
    assert ll.version().startswith("linear_layer_gb300")
    assert ll.status_string(ll.LL_ERR_WORKSPACE) == "LL_ERR_WORKSPACE"


def test_workspace_size_host_logic(built_lib):
    import linear_layer_gb300 as ll
    # aligned pitches need nothing
    assert ll.gemm_workspace_size(4096, 4096, 4096, 4096, 4096, ll.IN_BF16) == 0
    # FP16 ldb = 5003 -> 10006-byte pitch is not a multiple of 16: B (K x N) is repacked
    need = ll.gemm_workspace_size(4093, 5003, 2056, 2056, 5003, ll.IN_F16)
    assert need == 2056 * 10016 + 256
    # FP8 pitch 200 bytes is not a multiple of 16 either
    assert ll.gemm_workspace_size(10, 200, 64, 64, 200, ll.IN_E4M3) == 64 * 208 + 256
    assert ll.gemm_workspace_size(0, 5, 5, 5, 5, ll.IN_F16) == 0


def test_calls_without_a_gpu_fail_cleanly(built_lib):
    """A call that needs a device reports its absence instead of crashing (a call with no
    pointers, so nothing reaches a GPU even where one exists; the fake-address checks of
    every entry point run in a device-less child in test_abi_host_checks.py)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import linear_layer_gb300 as ll
    st = ll.lib.ll_get_device_status(None, None)
    assert st in (ll.LL_ERR_NO_DEVICE, ll.LL_ERR_CUDA)
    assert ll.lib.ll_set_wait_timeout_ns(1000) in (ll.LL_ERR_NO_DEVICE, ll.LL_ERR_CUDA)


def test_binding_refuses_host_tensors(built_lib):
    """A host tensor never reaches the library as a device pointer."""
    import torch
    import linear_layer_gb300 as ll
    host = torch.zeros(16, dtype=torch.int8)
    with pytest.raises(ValueError):
        ll.linear_w8a8_gemv(4, 16, host, host, host, 16, host, host)
    with pytest.raises(ValueError):
        ll.gemm_f16(1, 1, 1, 1.0, host, 1, host, 1, 0.0, None, 1, host, 1, ll.OUT_F32,
                    workspace=host)
