"""The benchmark's multi-rank path on CPU (gloo, world size 2): each rank
times its own batch; the step time is the maximum over ranks and the
whole-job throughput counts every rank's bytes (weak scaling)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [0.050 + 0.010 * rank, 0.170 - 0.020 * rank, 0.046 + 0.001 * rank]
        got = bench.max_over_ranks(mine, "cpu")
        value = bench.whole_job_gbs(world, 272891904.0, got[0])
        out.put((rank, got, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict()
    for _ in range(world):
        rank, got, value = q.get(timeout=120)
        results[rank] = (got, value)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    want = [0.060, 0.170, 0.047]
    for rank in range(world):
        got, value = results[rank]
        assert got == pytest.approx(want)
        # both ranks' bytes over the slowest rank's step
        assert value == pytest.approx(2 * 272891904.0 / (0.060e-3) / 1e9)


def test_whole_job_value_single_rank():
    import bench
    assert bench.whole_job_gbs(1, 272891904.0, 0.0474) == pytest.approx(272891904.0 / 47.4e-6 / 1e9)
