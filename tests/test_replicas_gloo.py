"""The multi-GPU path of the bench is independent replicas: each rank times
its own layer forwards, the job's time is the longest rank's, and the value
is that time over the units all ranks processed.  This host logic runs here
as two gloo ranks on the CPU (no GPU, no NCCL)."""
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


def _rank_main(rank, world, port, rank_ms, steps, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        dist.barrier()
        job_ms = bench.replica_max_ms(rank_ms[rank], "cpu")
        q.put((rank, r, w, local, job_ms, bench.per_unit_us(job_ms, steps, w)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_longest_rank_and_count_all_units():
    world, steps, rank_ms = 2, 100, [12.5, 20.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, rank_ms, steps, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, (r, rr, w, local, job_ms, us) in enumerate(got):
        assert (r, rr, w, local) == (rank, rank, world, rank)
        assert job_ms == max(rank_ms)  # every rank reports the job's time, the longest rank's
        assert us == pytest.approx(max(rank_ms) * 1e3 / (steps * world))  # units of both ranks


def test_single_process_is_its_own_job():
    import bench
    assert not dist.is_initialized()
    assert bench.replica_max_ms(7.25, "cpu") == 7.25
    assert bench.per_unit_us(7.25, 10, 1) == pytest.approx(725.0)

