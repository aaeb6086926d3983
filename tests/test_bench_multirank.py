"""The bench's multi-rank reduction on CPU: two gloo ranks, max over ranks of the step
times and the whole-job value (every rank's bytes over the slowest rank's time)."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step_ms, attn_ms = bench.max_over_ranks([1.0 + rank, 5.0 - rank], dist, "cpu")
        q.put((rank, step_ms, attn_ms, bench.job_gbs(world, 1e9, step_ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, step_ms, attn_ms, gbs in got:
        assert step_ms == 2.0 and attn_ms == 5.0  # the slowest rank's numbers on every rank
        assert gbs == pytest.approx(2 * 1e9 / 2e-3 / 1e9)


def test_single_rank_passthrough():
    import bench

    assert bench.max_over_ranks([3, 4]) == [3.0, 4.0]
    assert bench.job_gbs(1, 2e9, 1.0) == pytest.approx(2000.0)
