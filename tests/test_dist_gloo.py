"""The multi-rank host logic of bench.py (barrier, max over ranks, whole-job
throughput) on two CPU ranks with the gloo backend. Each rank of a real run is
an independent replica: no data crosses ranks, only these timing reductions."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    bench.barrier(world)
    ms = [3.0, 5.0][rank]  # the second rank is slower
    ms_max = bench.max_over_ranks(ms, world)
    value = bench.job_tokens_per_s(world, 32768, ms_max)
    q.put((rank, ms_max, value))
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms_max, value in got:
        assert ms_max == 5.0
        assert value == pytest.approx(2 * 32768 / 5e-3)
