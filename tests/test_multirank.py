"""Host logic of the data-parallel (replica) bench path on world_size 2 gloo ranks:
max-over-ranks timing, per-batch aggregation, and the reference arm printing on
rank 0 only."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 + 5 * rank, world)
        dist.barrier()
        q.put((rank, got, bench.per_batch_us(got, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
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
    assert [r[1] for r in res] == [15.0, 15.0]
    assert [r[2] for r in res] == [7500.0, 7500.0]   # 15 ms per step, 2 batches per step


def test_single_rank_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.per_batch_us(2.0, 1) == 2000.0


def test_reference_arm_silent_on_other_ranks():
    class A:
        config, seed, warmup, steps = 1, 0, 3, 1
    assert bench.run_reference(A, rank=1, world=2) is None
