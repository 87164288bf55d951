"""The multi-GPU path is replicas only (each rank runs its own layer on its
own tokens; nothing in the data path crosses ranks).  What crosses ranks is
the benchmark's timing: the slowest rank's step time, and the whole job's
tokens over it.  Checked here with two gloo ranks on the CPU."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        ms = [0.080, 0.095][rank]         # rank 1 is the slow one
        e2e = [0.120, 0.100][rank]
        out = bench.replica_throughput(ms, e2e, 2, ws, torch.device("cpu"))
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


def test_replica_throughput_takes_the_slowest_rank():
    ws, port = 2, 29500 + os.getpid() % 1000
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(ws):
        ms, ms_e2e, value, value_e2e = res[r]
        assert ms == pytest.approx(0.095) and ms_e2e == pytest.approx(0.120)
        assert value == pytest.approx(2 * 2 / 0.095e-3)       # both ranks' tokens over the slowest time
        assert value_e2e == pytest.approx(2 * 2 / 0.120e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ms, ms_e2e, value, value_e2e = bench.replica_throughput(0.5, 1.0, 8, 1, torch.device("cpu"))
    assert (ms, ms_e2e) == (0.5, 1.0) and value == pytest.approx(16000.0) and value_e2e == pytest.approx(8000.0)
