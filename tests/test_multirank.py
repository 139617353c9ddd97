"""Replicas on several ranks (host logic of bench.py under torchrun), on CPU with gloo:
each rank decodes its own cache; the job's step time is the max over ranks and the
throughput counts every rank's tokens.  The path has no collective on the data."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, ms, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench.dist_env()
        out.put((r, w, *bench.job_throughput(ms[rank], 8, world, "cpu")))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_job_throughput_takes_the_slowest_rank(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ms = [0.040, 0.052, 0.047][:world]
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, ms, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, w, job_ms, value) in enumerate(res):
        assert (r, w) == (rank, world)
        assert job_ms == pytest.approx(max(ms))
        assert value == pytest.approx(8 * world / (max(ms) / 1e3))


def test_single_rank_needs_no_process_group():
    import bench

    ms, value = bench.job_throughput(0.05, 8, 1)
    assert ms == 0.05 and value == pytest.approx(8 / 0.05e-3)
