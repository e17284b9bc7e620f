"""Host logic of bench.py's multi-GPU mode, run as two gloo ranks on the CPU:
the max-over-ranks reduction and the whole-job (weak-scaling) rate."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="env://")
    try:
        ws, r, local = bench.dist_env()
        local_ms = 10.0 + 5.0 * r  # rank r took 10 + 5r ms for its K steps
        slowest = bench.max_over_ranks(local_ms, ws)
        out.put((r, ws, local, slowest, bench.weak_rate(8192 * 4, slowest, ws)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_job_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = 10.0 + 5.0 * (world - 1)
    for r, (rank, ws, local, s, rate) in enumerate(got):
        assert (rank, ws, local) == (r, world, r)
        assert s == slowest
        # all ranks' samples over the slowest rank's time
        assert rate == pytest.approx(8192 * 4 * world / (slowest / 1e3))


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.weak_rate(100, 1000.0, 1) == pytest.approx(100.0)
