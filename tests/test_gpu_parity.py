"""CUDA path vs the CPU oracle, element by element, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from recsys_sparse_embedding_gb300 import binding, synth

from helpers import (TOL_BF16_EMUL, DeviceRun, assert_bf16_close, assert_f32_close, logits_of,
                     sample_ids)

pytestmark = pytest.mark.gpu

TC, F32 = binding.DSF_MODE_BF16_TC, binding.DSF_MODE_FP32


def check_batch(batch, samples=None, modes=(TC, F32), expect_status=0, check_logits=True,
                peaked=False):
    """peaked=True: logits are large, so bf16 rounding of the MLP operands moves
    the softmax far more than 2e-2 from the fp64 result; the bf16 path is then
    held to the oracle at the same operand precision only."""
    run = DeviceRun(batch)
    samples = np.arange(batch.B, dtype=np.int32) if samples is None else samples
    ref_pool, pflags = oracle.pool_batch(batch, samples)
    ref64, f64, lg64, _ = oracle.din_batch(batch, samples, want_logits=True)
    out = {}
    for mode in modes:
        pooled, din, lg, st = run.fwd(mode)
        assert st == expect_status, "status 0x%x" % st
        assert np.array_equal(pooled[samples], ref_pool), "pooled differs from the oracle"
        if mode == F32:
            if peaked:
                # fp32 rounding of large logits: |dz| ~ 2^-24 |z| moves the weights
                # by as much, so the bound grows with max|z| * max|s|
                zmax = np.abs(lg64[np.isfinite(lg64)]).max()
                smax = max(np.abs(t).max() for t in batch.tables)
                tol = 1e-5 + 16 * 2.0 ** -24 * zmax * smax
                assert np.abs(din[samples] - ref64).max() <= tol
            else:
                assert_f32_close(din[samples], ref64, "din fp32")
            print("fp32: max |din - fp64 oracle| = %.3e" % np.abs(din[samples] - ref64).max())
            if check_logits:
                g = logits_of(batch, samples, lg)
                m = np.isfinite(lg64)
                assert np.array_equal(np.isfinite(g), m)
                if peaked:
                    zmax = np.abs(lg64[m]).max()
                    assert np.abs(g[m] - lg64[m]).max() <= 1e-5 + 16 * 2.0 ** -24 * zmax
                else:
                    assert_f32_close(g[m], lg64[m], "logits fp32")
        else:
            emu, _, lge, _ = oracle.din_batch(batch, samples, bf16_mlp=True, want_logits=True)
            assert_bf16_close(din[samples], emu, "din bf16 vs bf16-operand oracle")
            if not peaked:
                assert_bf16_close(din[samples], ref64, "din bf16 vs fp64 oracle")
            err = np.abs(din[samples] - emu).max() if samples.size else 0.0
            print("bf16: max |din - bf16-operand oracle| = %.3e, max |din - fp64 oracle| = %.3e"
                  % (err, np.abs(din[samples] - ref64).max() if samples.size else 0.0))
            if not peaked:
                assert err <= TOL_BF16_EMUL, "din bf16 vs bf16-operand oracle: %.3e" % err
            if check_logits:
                g = logits_of(batch, samples, lg)
                m = np.isfinite(lge)
                assert np.array_equal(np.isfinite(g), m)
                zerr = np.abs(g[m] - lge[m])
                print("bf16: max |z - bf16-operand oracle z| = %.3e (max |z| %.2f)"
                      % (zerr.max() if zerr.size else 0.0, np.abs(lge[m]).max() if zerr.size else 0.0))
                if not peaked:
                    assert (zerr <= 2e-3 + 2e-3 * np.abs(lge[m])).all(), "logits bf16: %.3e" % zerr.max()
        out[mode] = (pooled, din)
    return run, out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_all_samples(seed):
    check_batch(synth.generate("tiny", seed=seed, nonzero_bias=True))


def test_tiny_peaked_softmax():
    check_batch(synth.generate("tiny", seed=3, peaked=True, nonzero_bias=True), peaked=True)


def test_tiny_page_table_map():
    check_batch(synth.generate("tiny", seed=4, seq_table=synth.SEQ_TABLES_PAGES))


@pytest.mark.parametrize("wl", ["taobao", "long_multihot"])
def test_small_batches_of_full_workloads(wl):
    # the workload's distributions at a batch the oracle finishes in seconds,
    # large enough for many CTAs, several tiles and ragged tails
    check_batch(synth.generate(wl, seed=1, B=1000, nonzero_bias=True))


def test_taobao_full_size_sampled():
    b = synth.generate("taobao", seed=0)
    check_batch(b, samples=sample_ids(b.B, 384))


def test_long_multihot_full_size_sampled():
    b = synth.generate("long_multihot", seed=0)
    check_batch(b, samples=sample_ids(b.B, 256))


def test_gather_stress_full_size_sampled():
    b = synth.generate("gather_stress", seed=0)
    check_batch(b, samples=sample_ids(b.B, 160), check_logits=False)


def test_wide_bf16_tables_both_modes():
    # D = 64: the tensor-core path streams W1 through the smem ring
    b = synth.generate("wide_bf16", seed=0, B=512, nonzero_bias=True)
    check_batch(b)


def test_wide_bf16_full_size_sampled():
    b = synth.generate("wide_bf16", seed=0)
    check_batch(b, samples=sample_ids(b.B, 160), check_logits=False)


def test_entry_points_agree():
    b = synth.generate("taobao", seed=2, B=3000, nonzero_bias=True)
    run = DeviceRun(b)
    for mode in (TC, F32):
        p_f, d_f, _, s1 = run.fwd(mode, "fused")
        p_p, _, _, s2 = run.fwd(mode, "pool")
        _, d_a, _, s3 = run.fwd(mode, "attn")
        assert s1 == s2 == s3 == 0
        assert np.array_equal(p_f, p_p)
        assert np.array_equal(d_f, d_a)


@pytest.mark.parametrize("wl,B,n", [("taobao", 20000, 512), ("long_multihot", 16384, 384),
                                     ("gather_stress", None, 256)])
def test_pool_only_large_batches(wl, B, n):
    # more than 64 samples per CTA batch: pooling alone takes four bags per thread
    b = synth.generate(wl, seed=1, B=B)
    run = DeviceRun(b)
    pooled, _, _, st = run.fwd(TC, "pool")
    assert st == 0, "status 0x%x" % st
    samples = sample_ids(b.B, n)
    ref_pool, _ = oracle.pool_batch(b, samples)
    assert np.array_equal(pooled[samples], ref_pool), "pooled differs from the oracle"


def test_repeated_calls_share_workspace():
    # the grid barrier resets itself between calls of different grid sizes
    b = synth.generate("tiny", seed=5, nonzero_bias=True)
    run = DeviceRun(b)
    first = run.fwd(TC)
    for i in range(20):
        which = ["fused", "pool", "attn"][i % 3]
        p, d, _, st = run.fwd(TC, which)
        assert st == 0
        if which != "attn":
            assert np.array_equal(p, first[0])
        if which != "pool":
            assert np.array_equal(d, first[1])


def _custom_batch(L, bags_len=None, max_len=100, D=16, rows=50, seed=0):
    rng = np.random.default_rng(seed)
    g = synth.generate("tiny", seed=seed, nonzero_bias=True)
    B, F = len(L), 16
    tables = [rng.standard_normal((rows, D)).astype(np.float32) * 0.05 for _ in range(F)]
    lengths = np.ones((F, B), np.int32) if bags_len is None else np.asarray(bags_len, np.int32)
    values = np.concatenate([rng.integers(0, rows, size=int(lengths[f].sum())) for f in range(F)])
    seq_lengths = np.asarray(L, np.int32)
    P = int(np.maximum(seq_lengths, 0).sum())
    seq_values = rng.integers(0, rows, size=(3, P)).astype(np.int64)
    return synth.Batch(wl=g.wl, B=B, tables=tables, lengths=lengths.reshape(-1),
                       values=values.astype(np.int64), seq_lengths=seq_lengths,
                       seq_values=seq_values, max_len=max_len, q_feat=(1, 5, 2),
                       seq_table=(1, 5, 2), W1=g.W1, b1=g.b1, W2=g.W2, b2=g.b2, w3=g.w3, b3=g.b3)


def test_edge_single_sample_and_empty_sequences():
    check_batch(_custom_batch([7]))
    check_batch(_custom_batch([0, 0, 0, 5, 0]))
    check_batch(_custom_batch([0] * 37))


def test_edge_long_sequences_span_tiles():
    # sequences longer than a 128-row tile, with a cap of 300: the softmax runs
    # online across tiles
    L = [250, 3, 129, 0, 300, 1, 128, 127]
    check_batch(_custom_batch(L, max_len=300))


def test_edge_truncation_flag():
    b = _custom_batch([120, 5, 101, 100], max_len=100)
    check_batch(b, expect_status=binding.FLAG_SEQ_TRUNC, check_logits=False)


def test_edge_empty_and_multi_hot_bags():
    rng = np.random.default_rng(3)
    lens = rng.integers(0, 6, size=(16, 300)).astype(np.int32)
    check_batch(_custom_batch(list(rng.integers(0, 20, size=300)), bags_len=lens))


def test_edge_out_of_range_ids_flagged_not_faulting():
    b = _custom_batch([4, 6, 3])
    b.values[3] = 10 ** 12
    b.values[5] = -7
    b.seq_values[1, 2] = 50           # == rows: out of range
    check_batch(b, expect_status=binding.FLAG_ID_RANGE)


def test_mean_pooling_deep_and_query_tables():
    """Mean-pooled tables, three of them query tables (1, 5, 2), so the
    attention's query is the bag mean too: the direct pooling path (bags of at
    most 16 values) on long_multihot, and the staged path on bags of up to 30."""
    pooling = tuple(1 if f in (0, 1, 2, 5, 9) else 0 for f in range(16))
    b = synth.generate("long_multihot", seed=0, B=1000)
    b.pooling = pooling
    check_batch(b, samples=sample_ids(b.B, 300))
    rng = np.random.default_rng(5)
    lens = rng.integers(0, 31, size=(16, 120)).astype(np.int32)
    c = _custom_batch(list(rng.integers(0, 40, size=120)), bags_len=lens)
    c.pooling = pooling
    check_batch(c)


def test_read_status_through_the_c_abi():
    """dsf_read_status returns the device word once the stream's earlier work
    is done: a flag a forward call sets, and a value written on a side stream."""
    b = _custom_batch([4, 6, 3])
    b.values[3] = 10 ** 12
    run = DeviceRun(b)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        binding.emb_bag_pool(run.db.tables, run.db.values, run.db.lengths, b.B,
                             torch.empty(b.B, b.F * b.D, device="cuda"), run.ws, status=st, stream=s)
    assert binding.read_status(st, stream=s) == binding.FLAG_ID_RANGE
    with torch.cuda.stream(s):
        st.fill_(0x1234)
    assert binding.read_status(st, stream=s) == 0x1234
