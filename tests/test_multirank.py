"""The benchmark's multi-GPU bookkeeping on CPU ranks (gloo, world size 2): each rank
times its own batch, the job's step time is the slowest rank's, and the throughput
counts every rank's tokens. The path itself shards by tokens with no data exchange."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [2.0, 3.5][rank]
    job_ms = bench.max_over_ranks(ms, world, torch.device("cpu"))
    q.put((rank, job_ms, bench.job_throughput(8192, world, job_ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_step_and_count_all_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, job_ms, value in res:
        assert job_ms == 3.5
        assert value == pytest.approx(2 * 8192 / 3.5e-3)


def test_single_rank_is_its_own_time():
    import bench
    assert bench.max_over_ranks(1.25, 1, torch.device("cpu")) == 1.25
    assert bench.job_throughput(64, 1, 0.5) == pytest.approx(128000.0)
