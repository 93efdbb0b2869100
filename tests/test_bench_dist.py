"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): replicas report
different elapsed times, the slowest rank's time is taken, whole-job throughput counts
every rank's work, and the oracle reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    bench.dist_init(world, "gloo")
    r, w, _ = bench.dist_env()
    t = bench.reduce_max(0.5 + r)  # rank r took 0.5 + r seconds
    value = bench.aggregate(100.0, w, t)
    bench.barrier()
    rc = bench.run_reference(bench.argparse.Namespace(steps=1, warmup=0)) if r == 1 else None
    q.put((r, w, t, value, rc))
    dist.destroy_process_group()


def test_two_rank_replicas_max_time_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, w, t, value, rc in res:
        assert w == 2
        assert t == pytest.approx(1.5)          # max over ranks
        assert value == pytest.approx(200.0 / 1.5)  # both ranks' units over the slowest time
    assert res[1][4] == 0  # the reference arm on rank 1 exits 0 without work


def test_single_process_helpers_without_process_group():
    import bench
    assert bench.reduce_max(3.25) == 3.25
    assert bench.aggregate(10.0, 1, 2.0) == 5.0
    assert bench.dist_env()[1] >= 1
