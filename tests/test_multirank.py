"""The N > 1 host path of bench.py on the CPU: world_size 2 over gloo (one
process per rank, rendezvous on 127.0.0.1).  The bench runs replicas -- the
path has no data exchange -- so what must hold is the timing rule: each
reported time is the maximum over ranks, and the value is the whole job's
throughput, world x (units per rank) / (slowest time)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r saw step time 1 + r ms and kernel time 10 - r ms
        ms, kms = bench.max_over_ranks([1.0 + rank, 10.0 - rank], torch.device("cpu"), world)
        dist.barrier()
        q.put((rank, ms, kms, bench.job_rate(1e6, ms, world)))
    finally:
        dist.destroy_process_group()


def test_replicas_time_is_max_over_ranks_and_value_is_whole_job():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, kms, rate in got:
        assert ms == 2.0 and kms == 10.0        # every rank holds the max of every time
        assert rate == pytest.approx(2 * 1e6 / 2e-3)  # world x units / slowest step


def test_single_rank_passes_through():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], torch.device("cpu"), 1) == [3.0, 4.0]
    assert bench.job_rate(5e6, 2.0, 1) == pytest.approx(2.5e9)
