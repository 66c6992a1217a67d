"""The bench's multi-rank logic on CPU: two gloo ranks report different timed-region
lengths; both must see the maximum, and the whole-job value counts every rank's step
(replicas, weak scaling)."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, torch.device("cpu"))
        out[rank] = ms
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_size_two():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_process_and_whole_job_value():
    import bench
    assert bench.max_over_ranks(12.5) == 12.5
    one = bench.whole_job_gbs(1, 357992576, 0.1567)
    assert abs(one - 357992576 / 0.1567e-3 / 1e9) < 1e-9
    assert abs(bench.whole_job_gbs(4, 357992576, 0.1567) - 4 * one) < 1e-9
