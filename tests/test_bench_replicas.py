"""bench.py's multi-process plumbing on CPU: barrier and max-over-ranks timing with gloo,
world size 2 (the GPU path runs the same calls over NCCL, one replica per GPU)."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_max = bench.max_over_ranks(1.5 + rank, world)
    bench.barrier(world)
    # weak scaling: every rank processes its own units; the job total uses the slowest rank
    units = 4 * world
    q.put((rank, ms_max, units / (ms_max / 1e3)))
    dist.destroy_process_group()


def test_two_rank_max_timing_and_weak_total():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5]              # every rank sees the max
    assert res[0][2] == pytest.approx(8 / 2.5e-3)         # 8 units over the slowest time
