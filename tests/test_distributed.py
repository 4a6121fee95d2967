"""Multi-rank bench logic on CPU with the gloo backend (world size 2).

bench.py runs N independent replicas of the layer, one per GPU (the layer
has no cross-GPU exchange); the job's step time is the maximum over ranks
and its throughput counts every rank's tokens.  This exercises that
aggregation over a real process group without a GPU.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step_ms, e2e_ms = 1.0 + rank, 5.0 - rank          # per-rank measurements
        mx = bench.reduce_max([step_ms, e2e_ms])
        q.put((rank, mx, bench.job_throughput(world, 8, mx[0]), bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, thr, env in got:
        assert mx == [2.0, 5.0]                  # max over ranks, element-wise
        assert thr == pytest.approx(2 * 8 / 2e-3)  # both ranks' tokens over the slowest step
        assert env == (rank, rank, 2)


def test_single_process_is_identity():
    assert bench.reduce_max([3.0, 4.0]) == [3.0, 4.0]
    assert bench.job_throughput(1, 8, 1.0) == pytest.approx(8000.0)
