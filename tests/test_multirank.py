"""The multi-GPU line is independent replicas (no data-path collective): the
host logic of bench.py's N > 1 path -- the job time is the slowest rank's, the
job throughput counts every rank's tokens, only rank 0 runs the reference arm --
checked with two gloo ranks on the CPU."""
import os
import socket
import sys
import types

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local_ms = 100.0 + 50.0 * rank           # rank 1 is the slower replica
        ms = bench.max_over_ranks(local_ms, dist, "cpu")
        value = bench.job_tokens_per_s(world, steps=10, tokens_per_step=1, ms=ms)
        args = types.SimpleNamespace(steps=1, warmup=0)
        ref = bench.bench_reference(args, None, world, rank, dist) if rank != 0 else "skipped"
        out.put((rank, ms, value, ref))
    finally:
        dist.destroy_process_group()


def test_two_replicas_max_time_and_total_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value, ref in res:
        assert ms == pytest.approx(150.0)                  # the slowest rank's time on every rank
        assert value == pytest.approx(2 * 10 * 1 / 0.150)  # both ranks' tokens over that time
        if rank == 1:
            assert ref is None                             # only rank 0 runs and prints the reference arm


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, None, "cpu") == 12.5
    assert bench.job_tokens_per_s(1, 4, 2, 1000.0) == pytest.approx(8.0)
