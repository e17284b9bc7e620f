"""Host logic of bench.py: the multi-GPU mode, run as two gloo ranks on the
CPU (the max-over-ranks reduction and the whole-job, weak-scaling rate), and
the JSON line of the reference arm."""
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


def test_reference_arm_prints_one_contract_line():
    # the reference arm is the CPU oracle: it runs without a GPU
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "samples/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
