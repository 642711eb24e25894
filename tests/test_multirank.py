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


def _ep_rank_main(rank, world, port, q):
    """One expert-parallel rank on CPU: its share of the tiny layer from the oracle (its
    half of the experts), the shares of all ranks through gather_partials (gloo), and
    their sum."""
    import datetime
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    import numpy as np
    import moe_inputs as mi
    import oracle
    from moe_expert_layer_count_gb300 import ep
    li = mi.make_layer_inputs(mi.TINY)
    E, per = li.wl.E, li.wl.E // world
    m = np.full(E, -1, np.int32)
    m[rank * per:(rank + 1) * per] = np.arange(per)
    sl = slice(rank * per, (rank + 1) * per)
    share = oracle.forward_chunked(li.x, li.topk_ids, li.topk_weights, li.w13[sl], li.w13_scale[sl], li.w2[sl],
                                   li.w2_scale[sl], E, expert_map=m)
    mine = torch.from_numpy(share.view(np.int16)).view(torch.bfloat16)
    parts = ep.gather_partials(mine)
    got = oracle.ep_combine([p.view(torch.int16).numpy().view(np.uint16) for p in parts])
    q.put((rank, got))
    dist.barrier()
    dist.destroy_process_group()


def test_expert_parallel_shares_gathered_over_two_ranks():
    """Two gloo ranks each hold half the experts; after gather_partials both hold both
    shares in rank order, and their sum is the single-rank layer within the layer
    tolerance (the same sum on both ranks)."""
    import numpy as np
    import moe_inputs as mi
    import oracle
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_ep_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        try:
            r, got = q.get(timeout=120)
        except Exception:
            break
        res[r] = got
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0, f"rank process exited with {p.exitcode}"
    assert sorted(res) == [0, 1]
    assert (res[0] == res[1]).all()
    li = mi.make_layer_inputs(mi.TINY)
    full = mi.bf16_to_f32(oracle.forward_chunked(li.x, li.topk_ids, li.topk_weights, li.w13, li.w13_scale, li.w2,
                                                 li.w2_scale, li.wl.E))
    got = mi.bf16_to_f32(res[0])
    err = np.abs(got - full)
    assert err.max() <= 2e-2 * np.abs(full).max() and err.sum() <= 5e-3 * np.abs(full).sum()
