"""The algorithmic byte and MAC counts the benchmark divides by, pinned to the batch-1
W8A8 example the A100 page prints ("NVIDIA A100: chip to SIMT", section 5.5: K = N =
4096 gives 16,777,216 useful INT8 MACs, a 16 MiB weight, a 4 KiB activation, a 16 KiB
FP32 per-output scale and an 8 KiB FP16 output)."""
import os

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "w8a8_example_scale.txt")


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = int(v)
    return vals


def test_gemv_bytes_match_the_printed_example():
    g = _golden()
    K, N = g["K"], g["N"]
    # weight + activation + per-output scales + output, plus the one FP32 activation scale
    printed = g["weight_bytes"] + g["activation_bytes"] + g["scale_bytes"] + g["output_bytes"]
    assert bench.gemv_bytes(N, K) == printed + 4


def test_useful_macs_match_the_printed_example():
    g = _golden()
    assert g["K"] * g["N"] == g["useful_macs"]
    # the GEMV's MACs are the weight bytes: every int8 weight is used once
    assert g["useful_macs"] == g["weight_bytes"]


def test_gemm_counts():
    # 2 M N K flops; A, B, C (FP32, read when beta != 0) and D bytes
    assert bench.gemm_flops(4096, 4096, 4096) == 2 * 4096 ** 3
    assert bench.gemm_bytes(4096, 4096, 4096, 2, 2, 1.0) == 167772160
    assert bench.gemm_bytes(256, 256, 256, 2, 4, 0.0) == 524288
