"""Row-wise sharded pooling (recsys_sparse_embedding_gb300.sharding) on two
gloo ranks on the CPU: each rank pools its half of the batch from tables
split by rows (and some whole on one rank), and its pooled rows must equal
the oracle's unsharded pooling of the same samples bit for bit. The pooling
primitive the sharded path calls is, in this CPU test, the oracle's pooling;
on GPUs it is the CUDA library's emb_bag_pool."""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SMALL_ROWS = [300_000, 150_000, 120_000, 9_000, 7_000, 5_000, 98, 14, 3, 8, 5, 5, 3, 7, 20, 40]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _np_table(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def oracle_pool(tables, values, lengths, B, pooling):
    """The pooling primitive, here the oracle's (pooled, flags)."""
    import oracle
    out, flags = oracle.emb_bag_pool([_np_table(t) for t in tables], values.numpy(), lengths.numpy(), B,
                                     None, pooling)
    return torch.from_numpy(out), int(flags)


def make_case(name):
    sys.path.insert(0, ROOT)
    from recsys_sparse_embedding_gb300 import synth
    if name == "taobao":
        b = synth.generate("taobao", seed=11, B=256, rows=SMALL_ROWS)
    elif name == "long_multihot":
        b = synth.generate("long_multihot", seed=12, B=200, rows=SMALL_ROWS)
        b.pooling = tuple(1 if f in (1, 3, 5) else 0 for f in range(16))
    elif name == "invalid_ids":
        b = synth.generate("long_multihot", seed=13, B=120, rows=SMALL_ROWS)
        b.values = np.array(b.values, copy=True)
        b.values[[0, 7, 400, 1000]] = [10 ** 9, -3, 300_000, 2 ** 40]
    elif name == "uniform_ids":
        b = synth.generate("gather_stress", seed=15, B=64, rows=SMALL_ROWS)
    elif name == "wide_bf16":
        b = synth.generate("wide_bf16", seed=14, B=96, rows=SMALL_ROWS)
    else:
        raise ValueError(name)
    return b


def local_kjt(b, lo, hi):
    """The KJT of samples [lo, hi): key-major values and lengths."""
    F, B = b.F, b.B
    lengths = np.maximum(np.asarray(b.lengths, np.int64).reshape(F, B), 0)
    off = np.concatenate([[0], np.cumsum(lengths.reshape(-1))])
    vals = []
    for f in range(F):
        vals.append(np.asarray(b.values)[off[f * B + lo]:off[f * B + hi]])
    return (np.concatenate(vals).astype(np.int64),
            np.asarray(b.lengths, np.int32).reshape(F, B)[:, lo:hi].reshape(-1).copy())


def _rank(rank, world, port, name, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from recsys_sparse_embedding_gb300 import sharding
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = make_case(name)
        bf = b.wl.dtype == "bf16"
        full = [torch.from_numpy(np.asarray(t)) for t in b.tables]
        if bf:
            full = [t.view(torch.bfloat16) for t in full]
        plan = sharding.ShardPlan.make([int(t.shape[0]) for t in full], world, row_wise_min_rows=100_000,
                                       table_wise=(3, 4))
        emb = sharding.RowWiseEmbeddingBag(plan, sharding.shard_tables(full, plan, rank), rank, oracle_pool,
                                           getattr(b, "pooling", None))
        per = -(-b.B // world)
        lo, hi = min(rank * per, b.B), min((rank + 1) * per, b.B)
        v, ln = local_kjt(b, lo, hi)
        pooled, flags = emb.forward(torch.from_numpy(v), torch.from_numpy(ln), hi - lo)
        held = sum(int(t.shape[0]) for t in emb.tables)
        q.put((rank, lo, hi, pooled.numpy(), flags, held, plan.kinds))
    finally:
        dist.destroy_process_group()


def run_ranks(name, world=2):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, name, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=300) for _ in range(world)), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return got


@pytest.mark.parametrize("name", ["taobao", "long_multihot", "invalid_ids", "uniform_ids", "wide_bf16"])
def test_row_wise_pooling_equals_unsharded_oracle(name):
    import oracle
    sys.path.insert(0, ROOT)
    b = make_case(name)
    got = run_ranks(name)
    ref_all, ref_flags = oracle.pool_batch(b)
    total_rows = sum(int(np.asarray(t).shape[0]) for t in b.tables)
    for rank, lo, hi, pooled, flags, held, kinds in got:
        assert pooled.shape == (hi - lo, b.F * b.D)
        assert np.array_equal(pooled, ref_all[lo:hi]), "rank %d pooled rows differ" % rank
        # the id-range flag where the rank's own samples hold such ids
        v, _ = local_kjt(b, lo, hi)
        bad = any(((v_f < 0) | (v_f >= n)).any() for v_f, n in _per_feature(b, v, lo, hi))
        assert bool(flags & 0x01) == bad
        # each rank holds about half of every row-wise table, not all of it
        assert held < total_rows
    assert kinds.count("row_wise") == 3 and kinds.count("table_wise") == 2
    if name == "invalid_ids":
        assert ref_flags & 0x01


def _per_feature(b, v, lo, hi):
    F, B = b.F, b.B
    lengths = np.maximum(np.asarray(b.lengths, np.int64).reshape(F, B)[:, lo:hi], 0)
    off = np.concatenate([[0], np.cumsum(lengths.sum(axis=1))])
    for f in range(F):
        yield v[off[f]:off[f + 1]], int(np.asarray(b.tables[f]).shape[0])


def test_plan_blocks_cover_every_row_once():
    sys.path.insert(0, ROOT)
    from recsys_sparse_embedding_gb300 import sharding
    for world in (1, 2, 3, 8):
        plan = sharding.ShardPlan.make([300_001, 100_000, 50, 7], world, row_wise_min_rows=100_000,
                                       table_wise=(3,))
        for f, n in enumerate(plan.rows):
            seen = np.zeros(n, np.int64)
            for r in range(world):
                lo, hi = plan.local_range(f, r)
                seen[lo:hi] += 1
            if plan.kinds[f] == "replicated":
                assert (seen == world).all()
            else:
                assert (seen == 1).all()
            ids = torch.tensor([0, n - 1, n, -1])
            own = plan.owner_of(f, ids).tolist() if plan.routed(f) else None
            if own is not None:
                assert own[2] == -1 and own[3] == -1
                for i, o in zip((0, n - 1), own[:2]):
                    lo, hi = plan.local_range(f, o)
                    assert lo <= i < hi


class ThreadExchange:
    """An in-process all-to-all for W ranks run as threads (host side only:
    the ranks' kernels never wait on one another)."""

    def __init__(self, world):
        import threading
        self.world = world
        self.bar = threading.Barrier(world)
        self.box = [None] * world

    def for_rank(self, rank):
        def ex(send, counts):
            self.box[rank] = (send, list(counts))
            self.bar.wait(timeout=60)
            parts, rcounts = [], []
            for src in range(self.world):
                s, c = self.box[src]
                a = sum(c[:rank])
                parts.append(s[a:a + c[rank]])
                rcounts.append(c[rank])
            self.bar.wait(timeout=60)
            return torch.cat(parts), rcounts
        return ex


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["long_multihot", "uniform_ids", "wide_bf16"])
def test_row_wise_pooling_on_the_gpu_two_emulated_ranks(name):
    """The same sharded pooling with the CUDA library as the pooling
    primitive, two ranks as threads of one process on one GPU exchanging
    through host code: pooled rows equal the oracle's bit for bit."""
    import threading
    import oracle
    sys.path.insert(0, ROOT)
    from recsys_sparse_embedding_gb300 import sharding
    b = make_case(name)
    world = 2
    full = [torch.from_numpy(np.asarray(t)) for t in b.tables]
    if b.wl.dtype == "bf16":
        full = [t.view(torch.bfloat16) for t in full]
    plan = sharding.ShardPlan.make([int(t.shape[0]) for t in full], world, row_wise_min_rows=100_000,
                                   table_wise=(3, 4))
    ex = ThreadExchange(world)
    ref, _ = oracle.pool_batch(b)
    out = [None] * world
    errs = []

    def rank_main(rank):
        try:
            torch.cuda.set_device(0)
            shards = [t.cuda() for t in sharding.shard_tables(full, plan, rank)]
            emb = sharding.RowWiseEmbeddingBag(plan, shards, rank, sharding.cuda_pool,
                                               getattr(b, "pooling", None), exchange=ex.for_rank(rank))
            per = -(-b.B // world)
            lo, hi = min(rank * per, b.B), min((rank + 1) * per, b.B)
            v, ln = local_kjt(b, lo, hi)
            pooled, flags = emb.forward(torch.from_numpy(v).cuda(), torch.from_numpy(ln).cuda(), hi - lo)
            out[rank] = (lo, hi, pooled.cpu().numpy(), flags)
        except Exception as e:  # reported below
            errs.append(e)
            ex.bar.abort()
    th = [threading.Thread(target=rank_main, args=(r,)) for r in range(world)]
    for t in th:
        t.start()
    for t in th:
        t.join(timeout=120)
    assert not errs, errs
    for lo, hi, pooled, flags in out:
        assert np.array_equal(pooled, ref[lo:hi])
