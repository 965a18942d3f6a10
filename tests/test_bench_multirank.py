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


def test_gpus_flag_starts_one_rank_per_gpu():
    """``bench.py --gpus 2`` run directly starts two ranks itself (through
    torch.distributed.run, rendezvous on 127.0.0.1) and rank 0 alone prints
    one line for the whole job. The reference arm runs on the host, so this
    needs no GPU: rank 0 times the oracle, rank 1 exits without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                       cwd=root, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    line = lines[0]
    assert line["n_gpus"] == 2 and line["impl"] == "reference" and line["steps"] == 1
    assert line["value"] > 0 and line["config"]["workload"].startswith("qwen3-8b layer")
