"""Hash-table (DynamicEmb-style) storage on the GPU, through the C ABI.

The tables above 100K rows are served by one hash table (independent key
spaces, one fused row pool, unseen keys read zero). The oracle resolves the
same raw keys by its own lookup (a sorted key list and a binary search), so
pooled rows are compared bit for bit and the attention output under the same
tolerances as the plain path."""
import numpy as np
import pytest
import torch

import oracle
from recsys_sparse_embedding_gb300 import binding, synth

from helpers import DeviceRun, sample_ids
from test_gpu_parity import F32, TC, _custom_batch, check_batch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cap", [1000, 600, 64])
def test_tiny_hashed_all_samples(cap):
    """All five large features hashed: every key admitted, 40% unseen, and
    nearly all unseen (only 64 rows admitted per table)."""
    b = synth.dynamic_emb(synth.generate("tiny", seed=cap, nonzero_bias=True), capacity=cap, seed=cap)
    check_batch(b)


def test_taobao_hashed_small_batch():
    """The pages' migration: five tables of 256K..1.14M ids, 300K admitted per
    table (the Zipf-hot ranks), the colder ids unseen."""
    b = synth.dynamic_emb(synth.generate("taobao", seed=1, B=1000, nonzero_bias=True), seed=1)
    check_batch(b)


def test_taobao_hashed_full_size_sampled():
    b = synth.dynamic_emb(synth.generate("taobao", seed=0), seed=0)
    check_batch(b, samples=sample_ids(b.B, 384))


def test_long_multihot_hashed_sampled():
    """Multi-hot bags (1..8 values) on exactly the hashed features."""
    b = synth.dynamic_emb(synth.generate("long_multihot", seed=2, B=2000, nonzero_bias=True), seed=2)
    check_batch(b, samples=sample_ids(b.B, 400))


def test_hashed_staged_pooling_and_mean():
    """Bags of up to 30 values (the staged pooling path) and mean pooling on
    hashed query tables: an unseen key adds a zero row and counts in the
    bag's length."""
    rng = np.random.default_rng(9)
    lens = rng.integers(0, 31, size=(16, 150)).astype(np.int32)
    c = _custom_batch(list(rng.integers(0, 40, size=150)), bags_len=lens, seed=9)
    c = synth.dynamic_emb(c, capacity=30, seed=9)
    check_batch(c)
    c.pooling = tuple(1 if f in (0, 1, 2, 7) else 0 for f in range(16))
    check_batch(c)


def test_hashed_entry_points_agree():
    b = synth.dynamic_emb(synth.generate("taobao", seed=2, B=3000, nonzero_bias=True), seed=2)
    run = DeviceRun(b)
    for mode in (TC, F32):
        p_f, d_f, _, s1 = run.fwd(mode, "fused")
        p_p, _, _, s2 = run.fwd(mode, "pool")
        _, d_a, _, s3 = run.fwd(mode, "attn")
        assert s1 == s2 == s3 == 0
        assert np.array_equal(p_f, p_p)
        assert np.array_equal(d_f, d_a)


def test_hashed_out_of_range_raw_keys_flagged():
    b = synth.dynamic_emb(synth.generate("tiny", seed=6, nonzero_bias=True), capacity=800, seed=6)
    b.values[3] = -5                    # feature 0
    b.values[64 + 7] = 1 << 60          # feature 1
    b.seq_values[0, 4] = -(1 << 62)     # adgroup sub-feature (hashed)
    check_batch(b, expect_status=binding.FLAG_ID_RANGE)


def _pool_single_ids(ht, table, keys, D=16):
    """pooled [n, D] of hashed table `table` (key space ht.key_space[table])
    whose n bags each hold one key; the other tables' bags are empty."""
    n = keys.numel()
    F = len(ht.key_space)
    dummy = torch.zeros(1, D, device="cuda")
    tabs = binding.EmbeddingTables([dummy] * F, None, ht)
    lengths = torch.zeros(F, n, dtype=torch.int32, device="cuda")
    lengths[table] = 1
    pooled = torch.full((n, F * D), float("nan"), device="cuda")
    ws = binding.Workspace(n, D)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.emb_bag_pool(tabs, keys, lengths.reshape(-1), n, pooled, ws, status=st)
    torch.cuda.synchronize()
    return pooled[:, table * D:(table + 1) * D].cpu().numpy(), int(st.item())


def test_insert_find_and_overwrite():
    rng = np.random.default_rng(1)
    n = 3000
    keys = np.unique(rng.integers(0, 1 << 56, size=n + 100))[:n]
    rows = (rng.standard_normal((n, 16)) * 0.05).astype(np.float32)
    ht = binding.HashTable(4096, 16, binding.DSF_F32, key_space=[3, 4])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kd = torch.from_numpy(keys).cuda()
    ht.insert(3, kd, torch.from_numpy(rows).cuda(), st)
    slots = ht.find(3, kd, st).cpu().numpy()
    assert int(st.item()) == 0
    n_slots = 4096
    assert np.unique(slots).size == n and slots.min() >= 0 and slots.max() < n_slots
    # another key space does not see these keys; unseen and invalid keys
    assert (ht.find(4, kd).cpu().numpy() == n_slots).all()
    unseen = torch.from_numpy(np.setdiff1d(rng.integers(0, 1 << 56, size=500), keys)).cuda()
    assert (ht.find(3, unseen).cpu().numpy() == n_slots).all()
    bad = torch.tensor([-1, 1 << 56, -(1 << 62)], dtype=torch.int64, device="cuda")
    st.zero_()
    assert ht.find(3, bad, st).cpu().numpy().tolist() == [-2, -2, -2]
    assert int(st.item()) == binding.FLAG_ID_RANGE
    # the rows behind the slots, read through the pooling path
    got, s = _pool_single_ids(ht, 0, torch.cat([kd, unseen]))
    assert s == 0
    assert np.array_equal(got[:n], rows) and not got[n:].any()
    # inserting present keys again overwrites their rows, in the same slots
    rows2 = rows[::-1].copy()
    ht.insert(3, kd, torch.from_numpy(rows2).cuda())
    assert np.array_equal(ht.find(3, kd).cpu().numpy(), slots)
    got2, _ = _pool_single_ids(ht, 0, kd)
    assert np.array_equal(got2, rows2)


def test_full_table_flags_and_keeps_what_fits():
    ht = binding.HashTable(8, 16, binding.DSF_F32, key_space=[0])   # one bucket of 8 slots
    keys = torch.arange(1000, 1020, dtype=torch.int64, device="cuda")
    rows = torch.randn(20, 16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ht.insert(0, keys, rows, st)
    assert int(st.item()) & binding.FLAG_HASH_FULL
    slots = ht.find(0, keys).cpu().numpy()
    held = slots < 8
    assert held.sum() == 8 and np.unique(slots[held]).size == 8


def test_uninitialised_workspace_flagged():
    b = synth.dynamic_emb(synth.generate("tiny", seed=8, B=16), capacity=1000, seed=8)
    run = DeviceRun(b)
    run.db.tables.hash.buf.zero_()      # header and keys gone: every probe sees full buckets
    _, _, _, st = run.fwd(TC)
    assert st & binding.FLAG_HASH


def test_wide_bf16_tables_hashed():
    """D = 64 bf16 rows in the hash pool (128-byte rows), both MLP modes."""
    b = synth.dynamic_emb(synth.generate("wide_bf16", seed=3, B=384, nonzero_bias=True), seed=3)
    check_batch(b)
