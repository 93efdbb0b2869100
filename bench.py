"""Benchmark of the linear-layer hot path on GB300.

Headline (one JSON line on rank 0): the BF16 GEMM M = N = K = 4096, alpha = 1,
beta = 1 (FP32 C), BF16 output, FP32 accumulation -- TFLOPS and its fraction of
the measured dense BF16 tensor peak.  A "step" is one call of the GEMM over one
batch of synthetic inputs already resident in HBM.  The same line carries the
other kernels of the path ("extra"): the batch-1 W8A8 GEMV 1 x 4096 . 4096 x 11008
(GB/s of HBM) and its fused FP16-activation form, the W8A8 and weight-only layers for a
few tokens, the FP8 E4M3 block-scaled GEMM 8192^3, the MXFP8 and NVFP4 GEMMs 8192^3
(hardware block scaling), the ragged FP16 GEMM 4093 x 5003 x 2056 and the launch-bound
FP16 256^3.  Every GEMM is given the workspace ll_gemm_*workspace_size asks for, so the
BF16 headline and the FP8 GEMM run their stream-K tails.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun): independent replicas, one per GPU, no data-path collective
(the path has no exchange step); value = work of all ranks / max-over-ranks time.
--impl reference times the CPU oracle on the host cores on a bounded sample of
the same workload (rank 0 only).
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOPS & % of GB300 dense tensor peak; W8A8 GEMV HBM GB/s & % of peak"
HEADLINE = "bf16_gemm_4096"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense FP8 : BF16 tensor throughput (4.5 : 2.25 PFLOP/s)
FP4_OVER_BF16 = 6.0  # nominal dense FP4 : BF16 tensor throughput (13.5 : 2.25 PFLOP/s)
L2_BYTES = 129 * 1000 * 1000
HEADLINE_GROUPS = 5  # the headline is the median of this many groups of `steps` steps

# algorithmic work per unit (one call) of each workload
def gemm_flops(M, N, K):
    return 2.0 * M * N * K


def gemm_bytes(M, N, K, in_bytes, out_bytes, beta):
    return M * K * in_bytes + K * N * in_bytes + (M * N * 4 if beta != 0 else 0) + M * N * out_bytes


def gemv_bytes(N, K):
    return N * K + K + 4 + 4 * N + 2 * N


KERNEL_SOURCES = {
    "gemm_mx_kernel": ["linear_layer_gb300/csrc/gemm_mx.cu", "linear_layer_gb300/csrc/gemm_common.cuh",
                       "linear_layer_gb300/csrc/ptx.cuh"],
    "gemm_mx2_kernel": ["linear_layer_gb300/csrc/gemm_mx.cu", "linear_layer_gb300/csrc/gemm_common.cuh",
                        "linear_layer_gb300/csrc/ptx.cuh"],
    "gemm_tc2_kernel": ["linear_layer_gb300/csrc/gemm_tc.cu", "linear_layer_gb300/csrc/gemm_common.cuh",
                        "linear_layer_gb300/csrc/ptx.cuh"],
    "gemm_tc_kernel": ["linear_layer_gb300/csrc/gemm_tc.cu", "linear_layer_gb300/csrc/gemm_common.cuh",
                       "linear_layer_gb300/csrc/ptx.cuh"],
    "gemv_w8a8_kernel": ["linear_layer_gb300/csrc/gemv_w8a8.cu", "linear_layer_gb300/csrc/ptx.cuh"],
}


def source_sha(kernel):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload, kernel):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("kernel") != kernel or rec.get("source_sha") != source_sha(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, ValueError, KeyError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def reduce_max(x, device=None):
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def aggregate(units_per_rank, world, max_seconds):
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="ll_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.15)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sms, maxes, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sms.append(float(parts[0]))
                    maxes.append(float(parts[1]))
                    power.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[4:8]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "power_w_max": max(power) if power else None, "samples": len(sms),
                "reasons": sorted(reasons)}


def gpu_smi_id(device_index):
    import torch
    try:
        uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[device_index]
        return device_index


# ------------------------------------------------------------------ our arm

def _up(a, dev):
    import numpy as np
    import torch
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def time_events(fn, steps, stream, per_call=True):
    """Run fn(i) for i < steps between two events on `stream`; with per_call, also time
    each call (an event between calls keeps consecutive kernels from overlapping, so
    the back-to-back timing leaves them out)."""
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    per = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)] if per_call else []
    start.record(stream)
    for i in range(steps):
        if per_call:
            per[i][0].record(stream)
        fn(i)
        if per_call:
            per[i][1].record(stream)
    end.record(stream)
    end.synchronize()
    total_ms = start.elapsed_time(end)
    launch_ms = [a.elapsed_time(b) for a, b in per]
    return total_ms, launch_ms


def bench_headline(args, dev, stream, rank, world, peaks, peak_src):
    import numpy as np
    import torch

    import linear_layer_gb300 as ll
    import workloads as wl
    cfg = wl.WORKLOADS[HEADLINE]
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    A, B, C = wl.gemm_inputs("bf16", M, N, K, cfg["beta"])
    set_bytes = gemm_bytes(M, N, K, 2, 2, cfg["beta"])
    nsets = max(2, math.ceil(4 * L2_BYTES / set_bytes))
    sets = []
    for _ in range(nsets):
        sets.append((_up(A, dev), _up(B, dev), _up(C, dev),
                     torch.empty((M, N), dtype=torch.bfloat16, device=dev)))

    # the workspace the library asks for (here: the partial tiles of its stream-K tail)
    ws_bytes = ll.gemm_workspace_size(M, N, K, K, N, ll.IN_BF16)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None

    def step(i):
        a, b, c, d = sets[i % nsets]
        ll.gemm_bf16(M, N, K, cfg["alpha"], a, K, b, N, cfg["beta"], c, N, d, N, ll.OUT_BF16,
                     workspace=ws, stream=stream)

    for i in range(args.warmup):
        step(i)
    st, word = ll.get_device_status(stream)
    if st != ll.LL_OK:
        raise RuntimeError("device status after warm-up: %s" % ll.status_string(st))
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(gpu_smi_id(dev.index))
    sampler.start()
    # HEADLINE_GROUPS groups of exactly `steps` steps, each bracketed by a barrier and a
    # synchronize and timed on the device; the reported group is the median one (max over
    # ranks within each group).  Steps within a group run back to back, as a model runs
    # its layers: programmatic dependent launch lets each GEMM's prologue overlap the
    # previous one's tail.
    group_s = []
    for _ in range(HEADLINE_GROUPS):
        barrier(dev)
        torch.cuda.synchronize(dev)
        total_ms, _ = time_events(step, args.steps, stream, per_call=False)
        torch.cuda.synchronize(dev)
        barrier(dev)
        group_s.append(reduce_max(total_ms / 1e3, dev))
    clocks = sampler.stop()
    st, word = ll.get_device_status(stream)
    if st != ll.LL_OK:
        raise RuntimeError("device status after timing: %s" % ll.status_string(st))
    max_s = statistics.median(group_s)
    total_ms = max_s * 1e3
    flops = gemm_flops(M, N, K)
    value = aggregate(flops * args.steps, world, max_s) / 1e12
    avg_launch_ms = total_ms / args.steps  # average launch duration over the median group
    achieved = flops / (avg_launch_ms / 1e3) / 1e12
    timed_s = total_ms / 1e3
    peak_key = "bf16_tflops_sustained" if timed_s > 2.0 else "bf16_tflops"
    peak = peaks[peak_key]
    roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": measured_traffic(HEADLINE, "gemm_tc2_kernel"),
                "kernel": "gemm_tc2_kernel<PairCfg<256>,9> (CTA pairs, BF16 x BF16)",
                "peak_source": "%s %s" % (peak_src, peak_key),
                "algorithmic_flops_per_launch": flops,
                "algorithmic_bytes_per_launch": set_bytes,
                "duration": "median group's timed region / steps (back-to-back launches)"}

    # end to end through the public API: every step copies its inputs A, B, C from pinned
    # host memory to the device, runs the GEMM and copies D back to pinned host memory.
    # Steps are pipelined over two device buffer sets: the copies of step i+1 (own
    # stream) overlap the GEMM of step i, and D of step i returns on a third stream.
    hA = torch.from_numpy(A.view(np.int16)).pin_memory()
    hB = torch.from_numpy(B.view(np.int16)).pin_memory()
    hC = torch.from_numpy(C).pin_memory()
    hD = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_mm = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = max(3, min(args.steps, 100))  # enough steps that pipeline fill and drain stay small

    def run_e2e(nsteps, t0=None, t1=None):
        if t0 is not None:
            t0.record(s_in)
        for i in range(nsteps):
            b = i % 2
            a, bb, c, d = sets[b]
            if i >= 2:
                s_in.wait_event(ev_mm[b])  # the GEMM of step i-2 is done with buffer b
            with torch.cuda.stream(s_in):
                a.copy_(hA, non_blocking=True)
                bb.copy_(hB, non_blocking=True)
                c.copy_(hC, non_blocking=True)
            ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # D of step i-2 has left buffer b
            ll.gemm_bf16(M, N, K, cfg["alpha"], a, K, bb, N, cfg["beta"], c, N, d, N, ll.OUT_BF16,
                         workspace=ws, stream=stream)
            ev_mm[b].record(stream)
            s_out.wait_event(ev_mm[b])
            with torch.cuda.stream(s_out):
                hD[b].copy_(d, non_blocking=True)
            ev_out[b].record(s_out)
        if t1 is not None:
            s_in.wait_stream(s_out)
            s_in.wait_stream(stream)
            t1.record(s_in)

    run_e2e(2)
    torch.cuda.synchronize(dev)
    barrier(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    run_e2e(e2e_steps, t0, t1)
    t1.synchronize()
    e2e_s = reduce_max(t0.elapsed_time(t1) / 1e3, dev)
    e2e = {"value": round(aggregate(flops * e2e_steps, world, e2e_s) / 1e12, 2), "unit": "TFLOPS",
           "h2d_bytes_per_step": int(hA.numel() * 2 + hB.numel() * 2 + hC.numel() * 4),
           "d2h_bytes_per_step": int(hD[0].numel() * 2), "steps": e2e_steps,
           "ms_per_step": round(e2e_s * 1e3 / e2e_steps, 4),
           "pipelining": "copies of step i+1 overlap the GEMM of step i (2 buffer sets, 3 streams)"}
    spread = {"groups": HEADLINE_GROUPS, "steps_per_group": args.steps,
              "ms_per_step_min_median_max": [round(min(group_s) * 1e3 / args.steps, 5),
                                             round(max_s * 1e3 / args.steps, 5),
                                             round(max(group_s) * 1e3 / args.steps, 5)],
              "tflops_min_max": [round(flops * args.steps / max(group_s) / 1e12, 1),
                                 round(flops * args.steps / min(group_s) / 1e12, 1)]}
    out = {"value": value, "ms_per_step": max_s * 1e3 / args.steps, "roofline": roofline,
           "e2e": e2e, "clocks": clocks, "gpu_launches": args.steps, "spread": spread,
           "config": {"workload": HEADLINE, "M": M, "N": N, "K": K, "alpha": cfg["alpha"],
                      "beta": cfg["beta"], "out": "bf16", "accumulate": "fp32",
                      "l2": "inputs rotate over %d resident sets (%.0f MB > L2)" % (
                          nsets, nsets * set_bytes / 1e6),
                      "workspace_bytes": ws_bytes,
                      "parallelism": "replicas" if world > 1 else "single"}}
    del sets
    return out


def bench_gemv(args, dev, stream, peaks, peak_src):
    import torch

    import linear_layer_gb300 as ll
    import workloads as wl
    cfg = wl.WORKLOADS["w8a8_gemv_4096x11008"]
    N, K = cfg["N"], cfg["K"]
    x, sx, W, sW = wl.gemv_inputs(N, K)
    wbytes = gemv_bytes(N, K)
    ncopies = max(2, math.ceil(4 * L2_BYTES / wbytes))
    tW0 = _up(W, dev)
    copies = []
    for _ in range(ncopies):
        copies.append((_up(x, dev), torch.tensor([sx], device=dev), tW0.clone(), _up(sW, dev),
                       torch.empty(N, dtype=torch.float16, device=dev)))
    del tW0

    def call(i):
        tx, tsx, tw, tsw, ty = copies[i % ncopies]
        ll.linear_w8a8_gemv(N, K, tx, tsx, tw, K, tsw, ty, None, stream=stream)

    for i in range(5):
        call(i)
    torch.cuda.synchronize(dev)
    per_graph = ncopies * 20
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for i in range(per_graph):
                call(i)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize(dev)
    reps = max(3, min(20, args.steps // 10 + 3))

    def replay(_):
        with torch.cuda.stream(stream):  # the graph launches on the current stream
            g.replay()

    total_ms, _ = time_events(replay, reps, stream)
    launch_s = total_ms / 1e3 / (reps * per_graph)
    gbs = wbytes / launch_s / 1e9
    peak = peaks["hbm_gbs"]
    # one launch at a time: an event on each side of every launch (which ends the overlap
    # with its neighbours), rotating over the weight copies so each launch streams from HBM
    _, single_ms = time_events(call, 50, stream, per_call=True)
    us_single = statistics.median(single_ms) * 1e3
    st, _ = ll.get_device_status(stream)
    return {"metric": "W8A8 GEMV HBM GB/s", "value": round(gbs, 1), "unit": "GB/s",
            "us_per_launch": round(launch_s * 1e6, 3),
            "us_single_launch": round(us_single, 3),
            "single_launch_GBs": round(wbytes / (us_single * 1e-6) / 1e9, 1),
            "single_launch_frac": round(wbytes / (us_single * 1e-6) / 1e9 / peak, 4),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4),
                         "traffic": measured_traffic("w8a8_gemv_4096x11008", "gemv_w8a8_kernel"),
                         "kernel": "gemv_w8a8_kernel", "peak_source": peak_src + " hbm_gbs",
                         "algorithmic_bytes_per_launch": wbytes},
            "timing": "CUDA graph of %d launches over %d weight copies (%.0f MB > L2), %d replays; "
                      "single launch: median of 50 launches with an event on each side" % (
                          per_graph, ncopies, ncopies * wbytes / 1e6, reps),
            "status": ll.status_string(st)}


def bench_gemv_fused(args, dev, stream, peaks, peak_src):
    """FP16 activation -> fused per-token quantiser + W8A8 GEMV + bias, FP16 out."""
    import numpy as np
    import torch

    import linear_layer_gb300 as ll
    import workloads as wl
    cfg = wl.WORKLOADS["w8a8_gemv_4096x11008"]
    N, K = cfg["N"], cfg["K"]
    _, _, W, sW = wl.gemv_inputs(N, K)
    xh = np.random.default_rng(wl.SEED_X).standard_normal(K).astype(np.float16)
    bias = np.random.default_rng(wl.SEED_C).standard_normal(N).astype(np.float32)
    wbytes = N * K + 2 * K + 4 * N + 4 * N + 2 * N + K + 4  # W, x fp16, s_W, bias, y, x_q, s_x
    ncopies = max(2, math.ceil(4 * L2_BYTES / wbytes))
    tW0 = _up(W, dev)
    copies = []
    for _ in range(ncopies):
        copies.append((torch.from_numpy(xh).to(dev), torch.empty(K, dtype=torch.int8, device=dev),
                       torch.empty(1, device=dev), tW0.clone(), _up(sW, dev), _up(bias, dev),
                       torch.empty(N, dtype=torch.float16, device=dev)))
    del tW0

    def call(i):
        tx, txq, txs, tw, tsw, tb, ty = copies[i % ncopies]
        ll.linear_f16_w8a8_gemv(N, K, tx, txq, txs, tw, K, tsw, tb, ll.GEMV_OUT_F16, None, ty,
                                stream=stream)

    for i in range(5):
        call(i)
    torch.cuda.synchronize(dev)
    per_graph = ncopies * 20
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for i in range(per_graph):
                call(i)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize(dev)
    reps = max(3, min(20, args.steps // 10 + 3))

    def replay(_):
        with torch.cuda.stream(stream):
            g.replay()

    total_ms, _ = time_events(replay, reps, stream)
    launch_s = total_ms / 1e3 / (reps * per_graph)
    gbs = wbytes / launch_s / 1e9
    peak = peaks["hbm_gbs"]
    st, _ = ll.get_device_status(stream)
    return {"metric": "FP16-activation W8A8 GEMV (fused per-token quantiser + bias) HBM GB/s",
            "value": round(gbs, 1), "unit": "GB/s", "us_per_launch": round(launch_s * 1e6, 3),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "traffic": None,
                         "kernel": "gemv_w8a8_kernel<true>", "peak_source": peak_src + " hbm_gbs",
                         "algorithmic_bytes_per_launch": wbytes},
            "timing": "CUDA graph of %d launches over %d weight copies, %d replays" % (
                per_graph, ncopies, reps),
            "status": ll.status_string(st)}


def bench_w8a8_tokens(args, dev, stream, peaks, peak_src):
    """The W8A8 layer (N = 11008, K = 4096) for a few tokens: dp4a up to 16 tokens, the
    exact FP16 tensor-core path in passes of up to 32 above that."""
    import torch

    import linear_layer_gb300 as ll
    import workloads as wl
    cfg = wl.WORKLOADS["w8a8_gemv_4096x11008"]
    N, K = cfg["N"], cfg["K"]
    out = {"metric": "W8A8 linear layer, several tokens: weight GB/s and int8 TOPS",
           "unit": "GB/s", "per_tokens": {}}
    _, _, W, sW = wl.batch_w8a8_inputs(1, N, K)
    ncopies = max(2, math.ceil(4 * L2_BYTES / (N * K)))
    tW0 = _up(W, dev)
    tWs = [tW0.clone() for _ in range(ncopies)]
    del tW0
    tsW = _up(sW, dev)
    for M in (2, 4, 8, 16, 24, 32):
        X, sx, _, _ = wl.batch_w8a8_inputs(M, N, K)
        tX, tsx = _up(X, dev), _up(sx, dev)
        tY = torch.empty((M, N), dtype=torch.float16, device=dev)

        def call(i):
            ll.linear_w8a8(M, N, K, tX, K, tsx, tWs[i % ncopies], K, tsW, None, ll.GEMV_OUT_F16, None,
                           tY, N, stream=stream)

        for i in range(5):
            call(i)
        torch.cuda.synchronize(dev)
        per_graph = ncopies * 20
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                for i in range(per_graph):
                    call(i)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
        torch.cuda.synchronize(dev)
        reps = max(3, min(20, args.steps // 10 + 3))

        def replay(_):
            with torch.cuda.stream(stream):
                g.replay()

        total_ms, _ = time_events(replay, reps, stream)
        launch_s = total_ms / 1e3 / (reps * per_graph)
        abytes = N * K + M * K + 4 * M + 4 * N + 2 * M * N
        out["per_tokens"][str(M)] = {
            "us_per_layer": round(launch_s * 1e6, 3),
            "GBs": round(abytes / launch_s / 1e9, 1),
            "frac_of_hbm": round(abytes / launch_s / 1e9 / peaks["hbm_gbs"], 4),
            "int8_TOPS": round(2.0 * M * N * K / launch_s / 1e12, 2),
            "path": "dp4a" if M <= 16 else "tensor cores (exact FP16 path)"}
        del g
    st, _ = ll.get_device_status(stream)
    out["value"] = out["per_tokens"]["2"]["GBs"]
    out["timing"] = "per token count: CUDA graph of %d launches over %d weight copies (%.0f MB > L2)" % (
        ncopies * 20, ncopies, ncopies * N * K / 1e6)
    out["status"] = ll.status_string(st)
    return out


def bench_w8a16(args, dev, stream, peaks, peak_src):
    """Weight-only INT8 layer with BF16 activations (N = 11008, K = 4096), 1..4 tokens."""
    import torch

    import linear_layer_gb300 as ll
    import workloads as wl
    cfg = wl.WORKLOADS["w8a8_gemv_4096x11008"]
    N, K = cfg["N"], cfg["K"]
    out = {"metric": "weight-only INT8 x BF16 linear layer: weight GB/s", "unit": "GB/s", "per_tokens": {}}
    _, W, sW = wl.w8a16_inputs(1, N, K)
    ncopies = max(2, math.ceil(4 * L2_BYTES / (N * K)))
    tW0 = _up(W, dev)
    tWs = [tW0.clone() for _ in range(ncopies)]
    del tW0
    tsW = _up(sW, dev)
    for M in (1, 2, 4):
        X, _, _ = wl.w8a16_inputs(M, N, K)
        tX = _up(X, dev)
        tY = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

        def call(i):
            ll.linear_w8a16(M, N, K, tX, K, tWs[i % ncopies], K, tsW, None, ll.OUT_BF16, tY, N, stream=stream)

        for i in range(5):
            call(i)
        torch.cuda.synchronize(dev)
        per_graph = ncopies * 20
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                for i in range(per_graph):
                    call(i)
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
        torch.cuda.synchronize(dev)
        reps = max(3, min(20, args.steps // 10 + 3))

        def replay(_):
            with torch.cuda.stream(stream):
                g.replay()

        total_ms, _ = time_events(replay, reps, stream)
        launch_s = total_ms / 1e3 / (reps * per_graph)
        abytes = N * K + 2 * M * K + 4 * N + 2 * M * N
        out["per_tokens"][str(M)] = {"us_per_layer": round(launch_s * 1e6, 3),
                                     "GBs": round(abytes / launch_s / 1e9, 1),
                                     "frac_of_hbm": round(abytes / launch_s / 1e9 / peaks["hbm_gbs"], 4)}
        del g
    st, _ = ll.get_device_status(stream)
    out["value"] = out["per_tokens"]["1"]["GBs"]
    out["timing"] = "per token count: CUDA graph of %d launches over %d weight copies" % (ncopies * 20, ncopies)
    out["status"] = ll.status_string(st)
    return out


def bench_fp8(args, dev, stream, peaks, peak_src):
    import torch

    import linear_layer_gb300 as ll
    import workloads as wl
    cfg = wl.WORKLOADS["e4m3_gemm_8192"]
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    A, sA, B, sB, _ = wl.fp8_inputs(M, N, K)
    tA, tsA, tB, tsB = _up(A, dev), _up(sA, dev), _up(B, dev), _up(sB, dev)
    sets = [(tA, tsA, tB, tsB, torch.empty((M, N), dtype=torch.bfloat16, device=dev))]
    sets.append((tA.clone(), tsA.clone(), tB.clone(), tsB.clone(),
                 torch.empty((M, N), dtype=torch.bfloat16, device=dev)))
    KB, NB = sA.shape[1], sB.shape[1]
    # the workspace the library asks for (here: the partial tiles of its stream-K tail)
    ws_bytes = ll.gemm_workspace_size(M, N, K, K, N, ll.IN_E4M3)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None

    def call(i):
        a, sa, b, sb, d = sets[i % 2]
        ll.gemm_fp8_blockscaled(M, N, K, 1.0, a, K, sa, KB, b, N, sb, NB, 0.0, None, N, d, N,
                                ll.OUT_BF16, workspace=ws, stream=stream)

    for i in range(3):
        call(i)
    torch.cuda.synchronize(dev)
    steps = max(10, min(args.steps // 10, 100))
    group_ms = []
    for _ in range(5):  # median of 5 groups of back-to-back launches
        total_ms, _ = time_events(call, steps, stream, per_call=False)
        group_ms.append(total_ms / steps)
    ms = statistics.median(group_ms)
    st, _ = ll.get_device_status(stream)
    flops = gemm_flops(M, N, K)
    tflops = flops / (ms / 1e3) / 1e12
    peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    return {"metric": "FP8 block-scaled GEMM TFLOPS", "value": round(tflops, 1), "unit": "TFLOPS",
            "ms_per_launch": round(ms, 4),
            "ms_per_launch_min_max": [round(min(group_ms), 4), round(max(group_ms), 4)],
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                         "traffic": measured_traffic("e4m3_gemm_8192", "gemm_tc_kernel"),
                         "kernel": "gemm_tc_kernel<TileCfg<256,true>,0> (one CTA per 128 x 256 tile)",
                         "peak_source": "%s bf16_tflops x %g (nominal FP8:BF16)" % (peak_src, FP8_OVER_BF16),
                         "algorithmic_bytes_per_launch": M * K + K * N + M * KB * 4 + KB * NB * 4 + M * N * 2},
            "timing": "median of 5 groups of %d back-to-back launches alternating 2 input sets "
                      "(A+B 128 MB each)" % steps,
            "workspace_bytes": ws_bytes,
            "status": ll.status_string(st)}


def bench_mx(args, dev, stream, peaks, peak_src):
    """MX block-scaled FP8 GEMM 8192^3 (E4M3, E8M0 scale per 32 K elements, BF16 out)."""
    import torch

    import linear_layer_gb300 as ll
    import workloads as wl
    cfg = wl.WORKLOADS["mxf8_gemm_8192"]
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    A, SA = wl.mx_quant(M, K, wl.SEED_A, 1)
    B, SB = wl.mx_quant(K, N, wl.SEED_B, 0)
    KB = SA.shape[1]
    tA, tSA, tB, tSB = _up(A, dev), _up(SA, dev), _up(B, dev), _up(SB, dev)
    sets = [(tA, tSA, tB, tSB, torch.empty((M, N), dtype=torch.bfloat16, device=dev))]
    sets.append((tA.clone(), tSA.clone(), tB.clone(), tSB.clone(),
                 torch.empty((M, N), dtype=torch.bfloat16, device=dev)))

    ws = torch.empty(ll.gemm_mxf8_workspace_size(M, N, K, K, N), dtype=torch.uint8, device=dev)

    def call(i):
        a, sa, b, sb, d = sets[i % 2]
        ll.gemm_mxf8(ll.IN_E4M3, ll.IN_E4M3, M, N, K, 1.0, a, K, sa, KB, b, N, sb, KB, 0.0, None, N, d, N,
                     ll.OUT_BF16, workspace=ws, stream=stream)

    for i in range(3):
        call(i)
    torch.cuda.synchronize(dev)
    steps = max(10, min(args.steps // 10, 100))
    group_ms = []
    for _ in range(5):  # median of 5 groups of back-to-back launches
        total_ms, _ = time_events(call, steps, stream, per_call=False)
        group_ms.append(total_ms / steps)
    ms = statistics.median(group_ms)
    st, _ = ll.get_device_status(stream)
    flops = gemm_flops(M, N, K)
    tflops = flops / (ms / 1e3) / 1e12
    peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    return {"metric": "MX block-scaled FP8 GEMM TFLOPS", "value": round(tflops, 1), "unit": "TFLOPS",
            "ms_per_launch": round(ms, 4),
            "ms_per_launch_min_max": [round(min(group_ms), 4), round(max(group_ms), 4)],
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                         "traffic": measured_traffic("mxf8_gemm_8192", "gemm_mx2_kernel"),
                         "kernel": "gemm_mx2_kernel<E4M3, MX> (CTA pairs per 256 x 256 tile, hardware block "
                                   "scaling)",
                         "peak_source": "%s bf16_tflops x %g (nominal FP8:BF16)" % (peak_src, FP8_OVER_BF16),
                         "algorithmic_bytes_per_launch": M * K + K * N + M * KB + N * KB + M * N * 2},
            "timing": "median of 5 groups of %d back-to-back calls alternating 2 input sets "
                      "(A+B 128 MB each); each call rearranges the scale codes, then runs the GEMM" % steps,
            "status": ll.status_string(st)}


def bench_nvf4(args, dev, stream, peaks, peak_src):
    """NVFP4 block-scaled GEMM 8192^3 (E2M1, UE4M3 scale per 16 K elements, BF16 out)."""
    import torch

    import linear_layer_gb300 as ll
    import workloads as wl
    cfg = wl.WORKLOADS["nvf4_gemm_8192"]
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    A, SA = wl.nvf4_quant(M, K, wl.SEED_A)
    Bt, SB = wl.nvf4_quant(N, K, wl.SEED_B)
    KB = SA.shape[1]
    tA, tSA, tB, tSB = _up(A, dev), _up(SA, dev), _up(Bt, dev), _up(SB, dev)
    # three input sets (A + Bt 64 MB each) and outputs (128 MB each): a set is read again
    # only after two other calls have moved 384 MB, three times L2
    sets = [(tA, tSA, tB, tSB, torch.empty((M, N), dtype=torch.bfloat16, device=dev))]
    for _ in range(2):
        sets.append((tA.clone(), tSA.clone(), tB.clone(), tSB.clone(),
                     torch.empty((M, N), dtype=torch.bfloat16, device=dev)))
    ws = torch.empty(ll.gemm_nvf4_workspace_size(M, N, K, K, K), dtype=torch.uint8, device=dev)

    def call(i):
        a, sa, b, sb, d = sets[i % 3]
        ll.gemm_nvf4(M, N, K, 1.0, a, K, sa, KB, b, K, sb, KB, 0.0, None, N, d, N, ll.OUT_BF16, workspace=ws,
                     stream=stream)

    for i in range(3):
        call(i)
    torch.cuda.synchronize(dev)
    steps = max(12, min(3 * (args.steps // 30), 120))
    group_ms = []
    for _ in range(5):  # median of 5 groups of back-to-back launches
        total_ms, _ = time_events(call, steps, stream, per_call=False)
        group_ms.append(total_ms / steps)
    ms = statistics.median(group_ms)
    st, _ = ll.get_device_status(stream)
    flops = gemm_flops(M, N, K)
    tflops = flops / (ms / 1e3) / 1e12
    peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    return {"metric": "NVFP4 block-scaled GEMM TFLOPS", "value": round(tflops, 1), "unit": "TFLOPS",
            "ms_per_launch": round(ms, 4),
            "ms_per_launch_min_max": [round(min(group_ms), 4), round(max(group_ms), 4)],
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": round(peak, 1),
                         "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                         "traffic": measured_traffic("nvf4_gemm_8192", "gemm_mx2_kernel"),
                         "kernel": "gemm_mx2_kernel<E2M1, NVFP4> (CTA pairs per 256 x 256 tile, hardware "
                                   "block scaling)",
                         "peak_source": "%s bf16_tflops x %g (nominal FP4:BF16)" % (peak_src, FP4_OVER_BF16),
                         "algorithmic_bytes_per_launch": M * K // 2 + N * K // 2 + M * KB + N * KB + M * N * 2},
            "timing": "median of 5 groups of %d back-to-back calls rotating 3 input sets "
                      "(A+Bt 64 MB each, D 128 MB each); each call rearranges the scale codes, then runs the "
                      "GEMM" % steps,
            "status": ll.status_string(st)}


def bench_small(args, dev, stream, peaks, peak_src):
    """FP16 256^3 with an FP32 output: launch-bound, so timed as a CUDA graph of 200
    launches; the roofline fraction is informational."""
    import torch

    import linear_layer_gb300 as ll
    import workloads as wl
    cfg = wl.WORKLOADS["f16_gemm_256"]
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    A, B, _ = wl.gemm_inputs("f16", M, N, K, cfg["beta"])
    tA, tB = _up(A, dev), _up(B, dev)
    tD = torch.empty((M, N), dtype=torch.float32, device=dev)

    def call(i):
        ll.gemm_f16(M, N, K, cfg["alpha"], tA, K, tB, N, cfg["beta"], None, N, tD, N, ll.OUT_F32,
                    stream=stream)

    for i in range(5):
        call(i)
    torch.cuda.synchronize(dev)
    per_graph = 200
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for i in range(per_graph):
                call(i)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize(dev)
    reps = 10

    def replay(_):
        with torch.cuda.stream(stream):
            g.replay()

    total_ms, _ = time_events(replay, reps, stream)
    launch_s = total_ms / 1e3 / (reps * per_graph)
    tflops = gemm_flops(M, N, K) / launch_s / 1e12
    peak = peaks["bf16_tflops"]
    st, _ = ll.get_device_status(stream)
    return {"metric": "FP16 GEMM 256^3 (launch-bound) time per launch", "value": round(launch_s * 1e6, 3),
            "unit": "us", "higher_is_better": False, "tflops": round(tflops, 2),
            "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tflops / peak, 5), "traffic": None,
                         "kernel": "gemm_tc_kernel (one CTA per 128-row tile)",
                         "peak_source": peak_src + " bf16_tflops (FP16 = BF16 rate); informational"},
            "timing": "CUDA graph of %d launches, %d replays; inputs (256 KB) stay in L2" % (per_graph, reps),
            "status": ll.status_string(st)}


def bench_ragged(args, dev, stream, peaks, peak_src):
    import torch

    import linear_layer_gb300 as ll
    import workloads as wl
    cfg = wl.WORKLOADS["f16_gemm_4093x5003x2056"]
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    A, B, C = wl.gemm_inputs("f16", M, N, K, cfg["beta"])
    tA, tB, tC = _up(A, dev), _up(B, dev), _up(C, dev)
    tD = torch.empty((M, N), dtype=torch.float32, device=dev)
    need = ll.gemm_workspace_size(M, N, K, K, N, ll.IN_F16)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)

    def call(i):
        ll.gemm_f16(M, N, K, cfg["alpha"], tA, K, tB, N, cfg["beta"], tC, N, tD, N, ll.OUT_F32,
                    workspace=ws, stream=stream)

    for i in range(3):
        call(i)
    torch.cuda.synchronize(dev)
    # median of 5 groups of back-to-back calls (one slow group does not set the figure)
    steps = max(5, min(args.steps // 50, 20))
    group_ms = []
    for _ in range(5):
        total_ms, _ = time_events(call, steps, stream, per_call=False)
        group_ms.append(total_ms / steps)
    ms = statistics.median(group_ms)
    st, _ = ll.get_device_status(stream)
    flops = gemm_flops(M, N, K)
    tflops = flops / (ms / 1e3) / 1e12
    peak = peaks["bf16_tflops"]
    return {"metric": "ragged FP16 GEMM TFLOPS (B repack of the 10006-byte pitch included)",
            "value": round(tflops, 1), "unit": "TFLOPS",
            "ms_per_call": round(ms, 4),
            "ms_per_call_min_max": [round(min(group_ms), 4), round(max(group_ms), 4)],
            "timing": "median of 5 groups of %d back-to-back calls" % steps,
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                         "traffic": measured_traffic("f16_gemm_4093x5003x2056", "gemm_tc2_kernel"),
                         "peak_source": peak_src + " bf16_tflops (FP16 = BF16 rate)"},
            "status": ll.status_string(st)}


def summarize(extra, head):
    """Short form of every workload's result: value, unit, roofline fraction, traffic."""
    out = {}
    for name, r in extra.items():
        e = {"value": r.get("value"), "unit": r.get("unit")}
        rf = r.get("roofline")
        if rf:
            e["frac"] = rf.get("frac")
            e["bound"] = rf.get("bound")
            e["peak"] = rf.get("peak")
            if rf.get("traffic") is not None:
                e["traffic"] = rf.get("traffic")
        for k in ("us_per_launch", "us_single_launch", "single_launch_frac", "ms_per_launch", "ms_per_call"):
            if k in r:
                e[k] = r[k]
        if "per_tokens" in r:
            e["per_tokens_GBs"] = {m: v["GBs"] for m, v in r["per_tokens"].items()}
        out[name] = e
    out["bf16_gemm_4096"] = {"value": round(head["value"], 1), "unit": "TFLOPS",
                             "frac": head["roofline"]["frac"],
                             "tflops_min_max": head["spread"]["tflops_min_max"]}
    return out


# ------------------------------------------------------------------ oracle (CPU) arm

def oracle_sample(target_s, min_rows=1):
    """Calibrate a sample of whole rows of the headline GEMM that the oracle computes in
    about target_s.  Returns (rows, run, cores, shape, last_seconds)."""
    import numpy as np

    import oracle
    import workloads as wl
    cfg = wl.WORKLOADS[HEADLINE]
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    A, B, C = wl.gemm_inputs("bf16", M, N, K, cfg["beta"])
    oracle.lib()

    def run(nrows):
        rows = np.linspace(0, M - 1, nrows).astype(np.int32)
        t0 = time.perf_counter()
        oracle.gemm("bf16", M, N, K, cfg["alpha"], A.ravel(), K, B.ravel(), N, cfg["beta"],
                    C.ravel(), N, rows=rows, want_absab=False)
        return time.perf_counter() - t0

    rows = max(min_rows, oracle.threads_used())
    t = run(rows)
    for _ in range(4):  # grow the sample until one run takes about target_s
        if t >= 0.8 * target_s or rows >= M:
            break
        rows = min(M, max(rows + 1, int(rows * target_s / max(t, 1e-3))))
        t = run(rows)
    return rows, run, oracle.threads_used(), (M, N, K), t


def cpu_baseline(target_s=12.0):
    rows, run, cores, (M, N, K), secs = oracle_sample(target_s)
    reps = 1
    if rows >= M and secs < 0.8 * target_s:  # the whole workload is shorter: repeat it
        reps = max(1, int(math.ceil(target_s / max(secs, 1e-3))))
        secs = sum(run(rows) for _ in range(reps))
    tflops = 2.0 * rows * N * K * reps / secs / 1e12
    return {"value": tflops, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
            "sample": "%d x %d of %d rows of the BF16 %dx%dx%d GEMM (double accumulation), %.1f s" % (
                reps, rows, M, M, N, K, secs)}


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    budget_s = 150.0
    per_step_s = budget_s / max(1, args.steps + args.warmup)
    rows, run, cores, (M, N, K), _ = oracle_sample(min(per_step_s, 10.0))
    for _ in range(args.warmup):
        run(rows)
    times = [run(rows) for _ in range(args.steps)]
    total = sum(times)
    value = 2.0 * rows * N * K * args.steps / total / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) BF16 A, B; FP32 C)",
            "config": {"workload": HEADLINE, "M": M, "N": N, "K": K, "alpha": 1.0, "beta": 1.0,
                       "out": "bf16", "sample_rows_per_step": rows},
            "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                             "sample": "%d of %d rows per step of the BF16 %dx%dx%d GEMM" % (rows, M, M, N, K)},
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ main

def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the GEMV / FP8 / ragged lines")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["all", "gemv", "gemv_fused", "fp8", "mx", "nvf4", "ragged", "tokens",
                                           "w8a16", "small"],
                    default="all",
                    help="all = the contract line; otherwise time one other kernel and print its object")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    rank, world, local = dist_env()
    import torch
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist_init(world, "nccl")
    import linear_layer_gb300 as ll  # fails loudly if the CUDA library is missing
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream(device=dev)

    single = {"gemv": bench_gemv, "gemv_fused": bench_gemv_fused, "fp8": bench_fp8, "mx": bench_mx,
              "nvf4": bench_nvf4, "ragged": bench_ragged, "tokens": bench_w8a8_tokens, "w8a16": bench_w8a16,
              "small": bench_small}.get(args.workload)
    if single is not None:
        res = single(args, dev, stream, peaks, peak_src)
        if rank == 0:
            print(json.dumps({"workload": args.workload, **res}), flush=True)
        return 0

    head = bench_headline(args, dev, stream, rank, world, peaks, peak_src)
    extra = {}
    if not args.no_extra:
        extra["w8a8_gemv_4096x11008"] = bench_gemv(args, dev, stream, peaks, peak_src)
        extra["f16_act_w8a8_gemv_fused_4096x11008"] = bench_gemv_fused(args, dev, stream, peaks,
                                                                       peak_src)
        extra["w8a8_linear_tokens_4096x11008"] = bench_w8a8_tokens(args, dev, stream, peaks, peak_src)
        extra["w8a16_linear_tokens_4096x11008"] = bench_w8a16(args, dev, stream, peaks, peak_src)
        extra["e4m3_gemm_8192"] = bench_fp8(args, dev, stream, peaks, peak_src)
        extra["mxf8_gemm_8192"] = bench_mx(args, dev, stream, peaks, peak_src)
        extra["nvf4_gemm_8192"] = bench_nvf4(args, dev, stream, peaks, peak_src)
        extra["f16_gemm_4093x5003x2056"] = bench_ragged(args, dev, stream, peaks, peak_src)
        extra["f16_gemm_256"] = bench_small(args, dev, stream, peaks, peak_src)
    barrier(dev)
    if rank != 0:
        return 0
    line = {"metric": METRIC, "value": round(head["value"], 2), "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(head["ms_per_step"], 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) BF16 A, B; FP32 C), resident in HBM",
            "config": head["config"], "roofline": head["roofline"], "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"], "clocks": head["clocks"], "spread": head["spread"],
            "library": ll.version(), "detail": extra}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    # the last key: one short entry per workload, so that the end of the line (what a log
    # tail keeps) carries every kernel's figure and roofline fraction
    line["extra"] = summarize(extra, head)
    print(json.dumps(line, separators=(",", ":")), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
