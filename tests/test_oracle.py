"""Pins for the CPU oracle: each test checks it against something other than
itself -- closed forms, exact integer sums, library routines, invariants and the
figures the pages print. No GPU needed."""
import dataclasses
import json
import math
import os

import numpy as np
import pytest

import oracle
from recsys_sparse_embedding_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers
def int_tables(rng, F, rows, D):
    """Integer-valued fp32 tables (|v| <= 64): every sum below is exact."""
    return [rng.integers(-64, 65, size=(rows, D)).astype(np.float32) for _ in range(F)]


def kjt_from_bags(bags, F, B):
    """bags[f][b] = list of ids -> key-major lengths / values."""
    lengths = np.array([len(bags[f][b]) for f in range(F) for b in range(B)], np.int32)
    values = np.array([i for f in range(F) for b in range(B) for i in bags[f][b]], np.int64)
    return lengths, values


def select_mlp(K1, col, scale, bias=10.0):
    """MLP whose logit is scale * (x[col] + bias) while x[col] + bias > 0:
    W1 row 0 picks x[col], W2 row 0 picks h1[0], w3 picks h2[0]."""
    W1 = np.zeros((256, K1), np.float32)
    W1[0, col] = 1.0
    b1 = np.zeros(256, np.float32)
    b1[0] = bias
    W2 = np.zeros((64, 256), np.float32)
    W2[0, 0] = 1.0
    b2 = np.zeros(64, np.float32)
    w3 = np.zeros(64, np.float32)
    w3[0] = scale
    b3 = np.zeros(1, np.float32)
    return W1, b1, W2, b2, w3, b3


def run_din(tables, lengths, values, B, seq_ids, seq_lengths, mlp, max_len=100,
            q_feat=(0, 1, 2), seq_table=(0, 1, 2), **kw):
    return oracle.din(tables, values, lengths, B, q_feat, seq_table, seq_ids, seq_lengths,
                      max_len, *mlp, **kw)


# ---------------------------------------------------------------- offsets
def test_offsets_all_ones_is_iota():
    n = 1000
    off, flags = oracle.offsets(np.ones(n, np.int32))
    assert flags == 0
    assert np.array_equal(off, np.arange(n + 1))


def test_offsets_hand_case_and_negative_flag():
    off, flags = oracle.offsets(np.array([2, 0, 3, 1], np.int32))
    assert list(off) == [0, 2, 2, 5, 6] and flags == 0
    off, flags = oracle.offsets(np.array([2, -4, 3], np.int32))
    assert list(off) == [0, 2, 2, 5] and flags == oracle.FLAG_NEG_LENGTH


# ---------------------------------------------------------------- pooling
def test_pool_single_id_bag_is_the_row():
    rng = np.random.default_rng(1)
    F, B, D = 4, 9, 16
    tables = [rng.standard_normal((50, D)).astype(np.float32) for _ in range(F)]
    ids = rng.integers(0, 50, size=(F, B))
    bags = [[[int(ids[f, b])] for b in range(B)] for f in range(F)]
    lengths, values = kjt_from_bags(bags, F, B)
    pooled, flags = oracle.emb_bag_pool(tables, values, lengths, B)
    assert flags == 0
    for b in range(B):
        for f in range(F):
            assert np.array_equal(pooled[b, f * D:(f + 1) * D], tables[f][ids[f, b]])


def test_pool_integer_tables_exact_and_permutation_invariant():
    rng = np.random.default_rng(2)
    F, B, D = 3, 17, 16
    tables = int_tables(rng, F, 40, D)
    bags = [[list(rng.integers(0, 40, size=rng.integers(0, 9))) for _ in range(B)]
            for _ in range(F)]
    lengths, values = kjt_from_bags(bags, F, B)
    pooled, flags = oracle.emb_bag_pool(tables, values, lengths, B)
    assert flags == 0
    for f in range(F):
        for b in range(B):
            want = np.zeros(D, np.int64)
            for i in bags[f][b]:
                want += tables[f][i].astype(np.int64)
            assert np.array_equal(pooled[b, f * D:(f + 1) * D], want.astype(np.float32))
    perm = [[list(rng.permutation(bags[f][b])) for b in range(B)] for f in range(F)]
    l2, v2 = kjt_from_bags(perm, F, B)
    pooled2, _ = oracle.emb_bag_pool(tables, v2, l2, B)
    assert np.array_equal(pooled, pooled2)


def test_pool_empty_bag_zero_and_out_of_range_flag():
    rng = np.random.default_rng(3)
    D = 16
    tables = [rng.standard_normal((10, D)).astype(np.float32) for _ in range(2)]
    bags = [[[], [3, 10]], [[-1], [2]]]    # empty bag; id 10 and -1 out of range
    lengths, values = kjt_from_bags(bags, 2, 2)
    pooled, flags = oracle.emb_bag_pool(tables, values, lengths, 2)
    assert flags == oracle.FLAG_ID_RANGE
    assert np.array_equal(pooled[0, :D], np.zeros(D, np.float32))
    assert np.array_equal(pooled[1, :D], tables[0][3])
    assert np.array_equal(pooled[0, D:], np.zeros(D, np.float32))
    assert np.array_equal(pooled[1, D:], tables[1][2])


def test_pool_fp32_sum_within_rounding_bound_of_exact_sum():
    """fp32 left-to-right sum of n terms is within n*eps*sum|terms| of the
    exact sum (here n <= 8, so well inside 1e-6 * sum|terms|)."""
    rng = np.random.default_rng(4)
    F, B, D = 2, 200, 16
    tables = [rng.standard_normal((100, D)).astype(np.float32) for _ in range(F)]
    bags = [[list(rng.integers(0, 100, size=rng.integers(1, 9))) for _ in range(B)]
            for _ in range(F)]
    lengths, values = kjt_from_bags(bags, F, B)
    pooled, _ = oracle.emb_bag_pool(tables, values, lengths, B)
    for f in range(F):
        for b in range(B):
            rows = tables[f][bags[f][b]].astype(np.float64)
            exact = rows.sum(0)
            bound = 1e-6 * np.abs(rows).sum(0)
            assert np.all(np.abs(pooled[b, f * D:(f + 1) * D] - exact) <= bound)


def test_pool_bf16_table_widens_exactly():
    rng = np.random.default_rng(5)
    D = 64
    t = synth.f32_to_bf16_bits(rng.standard_normal((30, D)).astype(np.float32))
    bags = [[[7], [29, 0]]]
    lengths, values = kjt_from_bags(bags, 1, 2)
    pooled, flags = oracle.emb_bag_pool([t], values, lengths, 2)
    assert flags == 0
    rows = synth.bf16_bits_to_f32(t)
    assert np.array_equal(pooled[0], rows[7])
    assert np.array_equal(pooled[1], (rows[29] + rows[0]).astype(np.float32))


# ---------------------------------------------------------------- MLP
def test_attn_mlp_matches_library_gemm():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((37, 192))
    b = synth.generate("tiny", seed=3, nonzero_bias=True)
    z = oracle.attn_mlp(x, b.W1, b.b1, b.W2, b.b2, b.w3, b.b3)
    W1, W2 = b.W1.astype(np.float64), b.W2.astype(np.float64)
    h1 = np.maximum(x @ W1.T + b.b1, 0)
    h2 = np.maximum(h1 @ W2.T + b.b2, 0)
    want = h2 @ b.w3.astype(np.float64) + b.b3[0]
    assert np.allclose(z, want, rtol=1e-12, atol=1e-12)


def test_attn_mlp_selection_closed_form():
    x = np.zeros((3, 192))
    x[:, 77] = [0.5, -2.0, 3.25]
    mlp = select_mlp(192, 77, scale=-1.5, bias=0.0)
    z = oracle.attn_mlp(x, *mlp)
    assert np.array_equal(z, -1.5 * np.maximum(x[:, 77], 0))


def test_attn_mlp_bf16_rounds_h1_to_nearest_even():
    # h1 = round_bf16(x + 0): 1 + 2^-8 is a tie -> 1; 1 + 3*2^-9 -> 1 + 2^-7
    x = np.zeros((2, 192))
    x[:, 5] = [1 + 2.0 ** -8, 1 + 3 * 2.0 ** -9]
    mlp = select_mlp(192, 5, scale=1.0, bias=0.0)
    z = oracle.attn_mlp(x, *mlp, bf16_mlp=True)
    assert list(z) == [1.0, 1 + 2.0 ** -7]


# ---------------------------------------------------------------- DIN
def tiny_din_inputs(rng, L_list, D=16, rows=20, positive=False):
    F, B = 3, len(L_list)
    lo = 0.05 if positive else -1.0
    tables = [rng.uniform(lo, 1.0, size=(rows, D)).astype(np.float32) for _ in range(F)]
    bags = [[[int(rng.integers(0, rows))] for _ in range(B)] for _ in range(F)]
    lengths, values = kjt_from_bags(bags, F, B)
    seq_lengths = np.array(L_list, np.int32)
    P = int(seq_lengths.sum())
    seq_ids = rng.integers(0, rows, size=(3, P)).astype(np.int64)
    return tables, lengths, values, seq_ids, seq_lengths, bags


def seq_rows(tables, seq_ids, seq_lengths, b, D=16):
    off = int(seq_lengths[:b].sum())
    L = int(seq_lengths[b])
    return np.stack([np.concatenate([tables[k][seq_ids[k, off + t]] for k in range(3)])
                     for t in range(L)]).astype(np.float64) if L else np.zeros((0, 3 * D))


def test_din_single_position_returns_that_row():
    rng = np.random.default_rng(7)
    t, l, v, sid, sl, _ = tiny_din_inputs(rng, [1, 1, 1])
    mlp = synth.generate("tiny", seed=1, nonzero_bias=True)
    out, flags = run_din(t, l, v, 3, sid, sl, (mlp.W1, mlp.b1, mlp.W2, mlp.b2, mlp.w3, mlp.b3))
    assert flags == 0
    for b in range(3):
        assert np.array_equal(out[b], seq_rows(t, sid, sl, b)[0])


def test_din_zero_w3_gives_mean_and_empty_gives_zero():
    rng = np.random.default_rng(8)
    t, l, v, sid, sl, _ = tiny_din_inputs(rng, [4, 0, 7])
    g = synth.generate("tiny", seed=2, nonzero_bias=True)
    mlp = (g.W1, g.b1, g.W2, g.b2, np.zeros(64, np.float32), g.b3)
    out, _ = run_din(t, l, v, 3, sid, sl, mlp)
    assert np.allclose(out[0], seq_rows(t, sid, sl, 0).mean(0), rtol=0, atol=1e-15)
    assert np.array_equal(out[1], np.zeros(48))
    assert np.allclose(out[2], seq_rows(t, sid, sl, 2).mean(0), rtol=0, atol=1e-15)


def test_din_identical_positions_return_the_row():
    rng = np.random.default_rng(9)
    t, l, v, sid, sl, _ = tiny_din_inputs(rng, [5])
    sid[:, :] = sid[:, :1]
    g = synth.generate("tiny", seed=4, nonzero_bias=True)
    out, _ = run_din(t, l, v, 1, sid, sl, (g.W1, g.b1, g.W2, g.b2, g.w3, g.b3))
    assert np.allclose(out[0], seq_rows(t, sid, sl, 0)[0], rtol=0, atol=1e-15)


@pytest.mark.parametrize("part", [0, 1, 2, 3])
def test_din_cat_order_two_positions_closed_form(part):
    """The input is cat[q, s, q - s, q * s]; with an MLP that selects one column
    of part `part`, two positions have softmax weight sigmoid(c*(x0 - x1))."""
    rng = np.random.default_rng(10 + part)
    t, l, v, sid, sl, bags = tiny_din_inputs(rng, [2], positive=True)
    d = 5
    c = 3.0
    mlp = select_mlp(192, part * 48 + d, scale=c, bias=10.0)
    out, flags = run_din(t, l, v, 1, sid, sl, mlp)
    assert flags == 0
    S = seq_rows(t, sid, sl, 0)
    q = np.concatenate([t[k][bags[k][0][0]] for k in range(3)]).astype(np.float64)
    xs = [q[d], S[:, d], q[d] - S[:, d], q[d] * S[:, d]][part]
    xs = np.broadcast_to(xs, (2,))
    a0 = 1.0 / (1.0 + math.exp(c * (xs[1] - xs[0])))
    want = a0 * S[0] + (1 - a0) * S[1]
    assert np.allclose(out[0], want, rtol=1e-13, atol=1e-15)


def test_din_query_is_the_pooled_multi_hot_bag():
    rng = np.random.default_rng(20)
    D, rows = 16, 20
    t = [rng.uniform(0.05, 1.0, size=(rows, D)).astype(np.float32) for _ in range(3)]
    bags = [[[1, 4, 9]], [[2]], [[3, 3]]]
    l, v = kjt_from_bags(bags, 3, 1)
    sl = np.array([2], np.int32)
    sid = rng.integers(0, rows, size=(3, 2)).astype(np.int64)
    d, c = 16 + 7, 2.0             # a column of the cate (second) block of q * s
    mlp = select_mlp(192, 3 * 48 + d, scale=c, bias=10.0)
    out, _ = run_din(t, l, v, 1, sid, sl, mlp)
    S = seq_rows(t, sid, sl, 0)
    qd = float(t[1][2][7])
    a0 = 1.0 / (1.0 + math.exp(c * qd * (S[1, d] - S[0, d])))
    assert np.allclose(out[0], a0 * S[0] + (1 - a0) * S[1], rtol=1e-13, atol=1e-15)
    # a multi-hot bag in the query: the q block of target 0 is the bag sum
    d0 = 3
    mlp = select_mlp(192, 3 * 48 + d0, scale=c, bias=10.0)
    out, _ = run_din(t, l, v, 1, sid, sl, mlp)
    q0 = float(np.float32(np.float32(t[0][1][3] + t[0][4][3]) + t[0][9][3]))
    a0 = 1.0 / (1.0 + math.exp(c * q0 * (S[1, d0] - S[0, d0])))
    assert np.allclose(out[0], a0 * S[0] + (1 - a0) * S[1], rtol=1e-13, atol=1e-15)


def test_din_padded_equals_jagged_bitwise():
    b = synth.generate("tiny", seed=5, nonzero_bias=True)
    jag, f1 = oracle.din_batch(b)
    pad, f2 = oracle.din_batch(b, padded=True)
    assert f1 == f2 == 0
    assert np.array_equal(jag, pad)
    jag, _ = oracle.din_batch(b, bf16_mlp=True)
    pad, _ = oracle.din_batch(b, padded=True, bf16_mlp=True)
    assert np.array_equal(jag, pad)


def test_din_weights_sum_to_one_and_permutation_invariance():
    b = synth.generate("tiny", seed=6, nonzero_bias=True, peaked=True)
    out, _, lg, wt = oracle.din_batch(b, want_logits=True)
    L = np.minimum(b.seq_lengths, b.max_len)
    for i in range(b.B):
        if L[i] > 0:
            assert abs(wt[i].sum() - 1.0) < 1e-12
            assert np.all(wt[i, L[i]:] == 0)
    # shuffle positions inside each sample
    rng = np.random.default_rng(0)
    off = np.concatenate([[0], np.cumsum(b.seq_lengths)])
    sv = b.seq_values.copy()
    for i in range(b.B):
        p = rng.permutation(b.seq_lengths[i]) + off[i]
        sv[:, off[i]:off[i + 1]] = sv[:, p]
    b2 = synth.Batch(**{**b.__dict__, "seq_values": sv})
    out2, _ = oracle.din_batch(b2)
    assert np.allclose(out, out2, rtol=0, atol=1e-14)


def test_din_peaked_softmax_picks_the_argmax_row():
    rng = np.random.default_rng(21)
    t, l, v, sid, sl, _ = tiny_din_inputs(rng, [6], positive=True)
    mlp = select_mlp(192, 48 + 2, scale=400.0, bias=10.0)   # z = 400 * s[2]
    out, _ = run_din(t, l, v, 1, sid, sl, mlp)
    S = seq_rows(t, sid, sl, 0)
    top = np.sort(S[:, 2])
    if top[-1] - top[-2] > 0.05:     # exp(-400*0.05) ~ 2e-9
        assert np.allclose(out[0], S[np.argmax(S[:, 2])], rtol=0, atol=1e-7)


def test_din_truncation_and_bad_ids():
    rng = np.random.default_rng(22)
    t, l, v, sid, sl, _ = tiny_din_inputs(rng, [5, 3])
    g = synth.generate("tiny", seed=7, nonzero_bias=True)
    mlp = (g.W1, g.b1, g.W2, g.b2, g.w3, g.b3)
    full, _ = run_din(t, l, v, 2, sid, sl, mlp, max_len=100)
    # max_len 3: sample 0 keeps its first 3 positions -- equal to a sample of length 3
    trunc, flags = run_din(t, l, v, 2, sid, sl, mlp, max_len=3)
    assert flags & oracle.FLAG_SEQ_TRUNC
    sid3 = np.concatenate([sid[:, :3], sid[:, 5:]], axis=1)
    ref, _ = run_din(t, l, v, 2, sid3, np.array([3, 3], np.int32), mlp, max_len=3)
    assert np.array_equal(trunc, ref)
    assert np.array_equal(trunc[1], full[1])
    # an out-of-range seq id gives a zero sub-row and the range flag
    sid_bad = sid.copy()
    sid_bad[1, 5] = 10 ** 9
    bad, flags = run_din(t, l, v, 2, sid_bad, sl, mlp)
    assert flags & oracle.FLAG_ID_RANGE
    assert np.array_equal(bad[0], full[0])


# ---------------------------------------------------------------- shapes
def test_workload_shapes_match_the_pages_figures():
    g = json.load(open(os.path.join(GOLDEN, "taobao_shapes.json")))
    rows = synth.TAOBAO_ROWS
    assert sum(rows[:15]) == g["id_feature_vocab_total"]["value"]
    mb = g["id_feature_vocab_total"]["value"] * g["embedding_dim"]["value"] * 4 / 2 ** 20
    assert round(mb) == g["embedding_weight_megabytes"]["value"]
    wl = synth.WORKLOADS["taobao"]
    assert wl.B == g["batch_size"]["value"] and wl.D == g["embedding_dim"]["value"]
    assert wl.max_len == g["sequence_cap"]["value"]
    assert wl.B * 5 * 3 * wl.D == g["seq_elements_real"]["value"]
    assert wl.B * wl.max_len * 3 * wl.D == g["seq_elements_padded"]["value"]
    assert wl.K1 == g["attention_input_width"]["value"]
    assert wl.Q == g["query_width"]["value"]
    assert [synth.ATTN_N1, synth.ATTN_N2] == g["attn_mlp_hidden"]["value"]


def test_generator_is_seeded_and_shaped():
    a = synth.generate("tiny", seed=11)
    b = synth.generate("tiny", seed=11)
    assert np.array_equal(a.values, b.values) and np.array_equal(a.seq_values, b.seq_values)
    assert a.lengths.size == 16 * 64 and a.values.size == a.lengths.sum()
    assert a.seq_values.shape == (3, a.seq_lengths.sum())
    assert a.seq_lengths.min() >= 0 and a.seq_lengths.max() <= 10


def test_mean_pooling_is_the_exact_mean_rounded_once():
    """EmbeddingBag mean mode (the pooling variant next to sum): each pooled
    element equals the exact rational mean of the bag's rows, rounded to the
    nearest float32. Integer-valued rows keep the fp32 sums exact, so the only
    rounding is the final division; the check compares against the exact mean
    with Fractions and the float32 neighbours of the result. Empty bags give 0;
    sum-pooled tables are untouched by the mode of the others."""
    from fractions import Fraction
    rng = np.random.default_rng(11)
    F, D, B, rows = 4, 16, 40, 30
    tables = [rng.integers(-64, 65, size=(rows, D)).astype(np.float32) for _ in range(F)]
    lengths = rng.integers(0, 9, size=(F, B)).astype(np.int32)
    values = np.concatenate([rng.integers(0, rows, size=int(lengths[f].sum())) for f in range(F)])
    pooling = np.array([1, 0, 1, 1], np.int32)
    got, flags = oracle.emb_bag_pool(tables, values, lengths.reshape(-1), B, pooling=pooling)
    summed, _ = oracle.emb_bag_pool(tables, values, lengths.reshape(-1), B)
    assert flags == 0
    off = np.concatenate([[0], np.cumsum(lengths.reshape(-1))])
    for f in range(F):
        for b in range(B):
            g = f * B + b
            ids = values[off[g]:off[g + 1]]
            cell = got[b, f * D:(f + 1) * D]
            if pooling[f] == 0:
                assert np.array_equal(cell, summed[b, f * D:(f + 1) * D])
                continue
            if ids.size == 0:
                assert np.all(cell == 0)
                continue
            for d in range(D):
                exact = Fraction(int(sum(int(tables[f][i, d]) for i in ids)), int(ids.size))
                r = np.float32(cell[d])
                lo = np.nextafter(r, np.float32(-np.inf))
                hi = np.nextafter(r, np.float32(np.inf))
                e = abs(Fraction(float(r)) - exact)
                assert e <= abs(Fraction(float(lo)) - exact) and e <= abs(Fraction(float(hi)) - exact), (f, b, d)


def _tower_zero():
    return dict(Wd1=np.zeros((512, 256), np.float32), bd1=np.zeros(512, np.float32),
                Wd2=np.zeros((256, 512), np.float32), bd2=np.zeros(256, np.float32),
                Wd3=np.zeros((128, 256), np.float32), bd3=np.zeros(128, np.float32),
                Wf1=np.zeros((64, 176), np.float32), bf1=np.zeros(64, np.float32),
                wo=np.zeros(64, np.float32), bo=np.zeros(1, np.float32))


def _towers(w, pooled, din, bf16=False):
    return oracle.towers(pooled, din, w["Wd1"], w["bd1"], w["Wd2"], w["bd2"], w["Wd3"], w["bd3"],
                         w["Wf1"], w["bf1"], w["wo"], w["bo"], bf16_mlp=bf16)


def test_towers_zero_weights_give_the_bias_path():
    """All weight matrices zero: y = b_o + w_o . ReLU(b_f1), whatever the inputs
    (the deep tower then feeds ReLU(b_d3) forward, which W_f1 = 0 ignores)."""
    rng = np.random.default_rng(21)
    w = _tower_zero()
    w["bf1"][:] = rng.uniform(-1, 1, 64)
    w["wo"][:] = rng.uniform(-1, 1, 64)
    w["bo"][:] = 0.25
    pooled = rng.standard_normal((7, 256)).astype(np.float32)
    din = rng.standard_normal((7, 48))
    want = 0.25 + float(np.dot(w["wo"].astype(np.float64), np.maximum(w["bf1"].astype(np.float64), 0)))
    for bf16 in (False, True):
        y = _towers(w, pooled, din, bf16)
        assert np.allclose(y, want, rtol=0, atol=1e-12)


def test_towers_identity_chain_is_the_mean_of_the_final_input():
    """Non-negative inputs through identity blocks (Linear [out, in]: W_d1 = [I; 0],
    W_d2 = [I 0], W_d3 = [I 0], zero biases) reach the final tower as
    cat[p[:128], din]; one row of W_f1 = 1/176 then gives its mean: y equals
    (sum p[:128] + sum din) / 176 exactly up to rounding. A transposed weight,
    a shifted slice or a swapped cat order changes the value."""
    rng = np.random.default_rng(22)
    w = _tower_zero()
    w["Wd1"][:256, :] = np.eye(256, dtype=np.float32)
    w["Wd2"][:, :256] = np.eye(256, dtype=np.float32)
    w["Wd3"][:, :128] = np.eye(128, dtype=np.float32)
    w["Wf1"][0, :] = 1.0 / 176
    w["wo"][0] = 1.0
    pooled = rng.uniform(0, 1, (9, 256)).astype(np.float32)
    din = rng.uniform(0, 1, (9, 48))
    want = (pooled[:, :128].astype(np.float64).sum(1) + din.sum(1)) / 176
    y = _towers(w, pooled, din)
    assert np.allclose(y, want, rtol=1e-6, atol=0)
    # a single din slot: W_f1 row 0 picks position 128 + 5 of cat[h, din]
    w["Wf1"][0, :] = 0.0
    w["Wf1"][0, 128 + 5] = 1.0
    assert np.allclose(_towers(w, pooled, din), din[:, 5], rtol=0, atol=1e-15)


def test_towers_relu_after_every_hidden_layer():
    """W_d1 = -[I; 0]: the first layer's pre-activations are -p <= 0 for p >= 0,
    so ReLU zeroes them and the rest sees h1 = 0: y = b_o + w_o . ReLU(W_f1
    cat[ReLU(b_d3), din] + b_f1) with b_d2 = 0, here with W_f1 picking b_d3's
    first slot (kept by ReLU) and a negative b_f1 entry (cut by ReLU)."""
    w = _tower_zero()
    w["Wd1"][:256, :] = -np.eye(256, dtype=np.float32)
    w["bd3"][0] = 0.5
    w["Wf1"][0, 0] = 2.0
    w["bf1"][1] = -3.0
    w["wo"][:2] = (1.0, 1.0)
    pooled = np.abs(np.random.default_rng(23).standard_normal((4, 256))).astype(np.float32)
    y = _towers(w, pooled, np.zeros((4, 48)))
    assert np.allclose(y, 1.0, rtol=0, atol=1e-15)   # 2 * 0.5 + ReLU(-3) = 1


def test_towers_bf16_mode_is_exact_on_bf16_representable_data():
    """Inputs, weights and every intermediate exactly representable in bf16
    (small multiples of 1/8 through identity-like layers): the bf16-operand
    mode and the double mode agree to the last bit."""
    rng = np.random.default_rng(24)
    w = _tower_zero()
    w["Wd1"][:256, :] = np.eye(256, dtype=np.float32)
    w["Wd2"][:, :256] = np.eye(256, dtype=np.float32)
    w["Wd3"][:, :128] = np.eye(128, dtype=np.float32)
    w["Wf1"][np.arange(64), np.arange(64) * 2] = 1.0
    w["wo"][:] = 0.5
    pooled = (rng.integers(0, 16, (6, 256)) / 8).astype(np.float32)
    din = rng.integers(0, 16, (6, 48)) / 8.0
    assert np.array_equal(_towers(w, pooled, din), _towers(w, pooled, din, True))


# ---------------------------------------------------------------- hash tables
def test_hash_translate_matches_a_dict():
    """The lookup against a brute-force dict: admitted keys read their own
    row, unseen keys the appended zero row, keys outside [0, 2^56) are -1."""
    rng = np.random.default_rng(7)
    keys = np.unique(rng.integers(0, 1 << 56, size=3000))[:2000]
    keys = rng.permutation(keys)
    row_of = {int(k): i for i, k in enumerate(keys)}
    q = np.concatenate([rng.choice(keys, 500), rng.integers(0, 1 << 56, size=500),
                        np.array([-1, -(1 << 40), 1 << 56, (1 << 63) - 1, 0])])
    want = [(-1 if (x < 0 or x >= 1 << 56) else row_of.get(int(x), keys.size)) for x in q]
    assert oracle.hash_translate(keys, q).tolist() == want
    assert oracle.hash_translate(np.zeros(0, np.int64), np.array([5])).tolist() == [0]


def _zero_cold_rows(plain, cap, feats):
    """The plain batch with every row at or above `cap` of `feats` zeroed:
    what a table that admitted only the first `cap` rows returns."""
    tables = [t.copy() for t in plain.tables]
    for f in feats:
        tables[f][cap:] = 0
    return dataclasses.replace(plain, tables=tables)


@pytest.mark.parametrize("cap", [1000, 600, 1])
def test_hashed_batch_equals_plain_batch_with_cold_rows_zeroed(cap):
    """Hash-table features give exactly the plain path's pooled rows and DIN
    output once the rows the table did not admit read as zero."""
    plain = synth.generate("tiny", seed=3, nonzero_bias=True)
    hashed = synth.dynamic_emb(plain, capacity=cap, seed=3)
    ref = _zero_cold_rows(plain, cap, synth.DYNEMB_FEATURES)
    p_h, fl_h = oracle.pool_batch(hashed)
    p_r, fl_r = oracle.pool_batch(ref)
    assert fl_h == fl_r == 0
    assert np.array_equal(p_h, p_r)
    d_h, _ = oracle.din_batch(hashed)
    d_r, _ = oracle.din_batch(ref)
    assert np.array_equal(d_h, d_r)
    if cap < 1000:  # some ids are unseen, so the cold rows mattered
        assert not np.array_equal(p_r, oracle.pool_batch(plain)[0])


def test_hash_key_spaces_of_different_tables_are_independent():
    """One raw key admitted by two tables reads each table's own row; a key
    admitted only by table 0 is unseen (zero) in table 1."""
    plain = synth.generate("tiny", seed=4, B=8)
    hashed = synth.dynamic_emb(plain, features=(0, 1), capacity=1000, seed=4)
    k0, k1 = hashed.hash_keys[0].copy(), hashed.hash_keys[1].copy()
    k1[7] = k0[3]          # the same raw key, rows 3 of table 0 and 7 of table 1
    shared, only0 = k0[3], k0[5]
    assert only0 not in set(k1.tolist())
    hk = {0: k0, 1: k1}
    B = hashed.B
    vals = hashed.values.copy()
    vals[0] = shared       # sample 0 of feature 0
    vals[B] = shared       # sample 0 of feature 1
    vals[B + 1] = only0    # sample 1 of feature 1
    b = dataclasses.replace(hashed, hash_keys=hk, values=vals)
    pooled, _ = oracle.pool_batch(b)
    D = b.D
    assert np.array_equal(pooled[0, 0:D], b.tables[0][3])
    assert np.array_equal(pooled[0, D:2 * D], b.tables[1][7])
    assert not pooled[1, D:2 * D].any()


# ---------------------------------------------------------------- backward
from oracle import backward as obw  # noqa: E402


def _small_batch(seed=0, B=6, rows=12, f64=False, wl="long_multihot"):
    """A small batch with few rows per table, so rows repeat across bags,
    features and positions; bags of 1..8 values on features 0-4; nonzero
    biases."""
    g = synth.generate(wl, seed=seed, B=B, rows=[rows] * 16, nonzero_bias=True)
    if f64:
        g = dataclasses.replace(g, tables=[t.astype(np.float64) for t in g.tables])
    return g


@pytest.mark.parametrize("bf16", [False, True])
def test_backward_forward_equals_oracle_din(bf16):
    """The backward oracle's own forward reproduces oracle_din (fp64 and the
    bf16-operand mode) on a workload batch."""
    b = synth.generate("tiny", seed=2, nonzero_bias=True)
    ref, _ = oracle.din_batch(b, bf16_mlp=bf16)
    fw = obw.forward(b, bf16)
    assert np.abs(fw["din"] - ref).max() <= 1e-12


def test_backward_matches_finite_differences():
    """Every gradient against central differences of the fp64 forward on
    loss = sum(dpooled * pooled) + sum(ddin * din): table rows reached through
    deep bags, the query and the sequence, and entries of every MLP tensor."""
    b = _small_batch(seed=1, f64=True)
    b.pooling = tuple(1 if f in (1, 3) else 0 for f in range(16))  # multi-hot query and plain tables by mean
    rng = np.random.default_rng(0)
    B, F, D = b.B, b.F, b.D
    dpooled = rng.standard_normal((B, F * D))
    ddin = rng.standard_normal((B, 3 * D))

    def loss(bb):
        fw = obw.forward(bb)
        return float((dpooled * obw.pooled64(bb)).sum() + (ddin * fw["din"]).sum())
    g = obw.backward(b, dpooled, ddin)
    h = 1e-6

    def fd(mutate):
        return (loss(mutate(+h)) - loss(mutate(-h))) / (2 * h)

    def check(an, num):
        assert abs(an - num) <= 1e-6 * max(1.0, abs(num)), (an, num)
    # table rows: one of a query table (1), of a plain deep table (7), of a
    # sequence-only lookup through table 2
    for f in (1, 2, 3, 7):
        rows, grads = g["rows"][f]
        for ri in (0, len(rows) - 1):
            r, d = int(rows[ri]), 3

            def mut(e, f=f, r=r, d=d):
                tabs = [t.copy() for t in b.tables]
                tabs[f][r, d] += e
                return dataclasses.replace(b, tables=tabs)
            check(grads[ri, d], fd(mut))
    for name, idx in (("W1", (5, 17)), ("W1", (200, 150)), ("b1", (3,)), ("W2", (7, 100)),
                      ("b2", (11,)), ("w3", (9,)), ("b3", (0,))):
        def mut(e, name=name, idx=idx):
            a = getattr(b, name).astype(np.float64).copy()
            a[idx] += e
            return dataclasses.replace(b, **{name: a})
        an = g["d" + name][idx] if name != "b3" else g["db3"][0]
        check(an, fd(mut))


def test_backward_bf16_operands_stay_within_bf16_error():
    """The bf16-operand mode differs from fp64 only through the roundings of
    the GEMM operands (2^-9 relative each), measured against the sum of each
    gradient entry's term magnitudes. (Relative to the entry itself the
    difference can be large: per sample the dz_t sum to zero, so the
    gradients are small residuals of larger terms.)"""
    b = synth.generate("tiny", seed=3, nonzero_bias=True)
    rng = np.random.default_rng(1)
    ddin = rng.standard_normal((b.B, 3 * b.D))
    g64 = obw.backward(b, None, ddin)
    g16 = obw.backward(b, None, ddin, bf16=True)
    fw = obw.forward(b)
    a, s = fw["a"], fw["s32"].astype(np.float64)
    samp = fw["samp"]
    da = np.einsum("pd,pd->p", ddin[samp], s)
    c = np.zeros(b.B)
    np.add.at(c, samp, a * da)
    dz = a * (da - c[samp])
    dh2 = np.abs(dz)[:, None] * np.abs(b.w3)[None, :]
    dh1 = dh2 @ np.abs(b.W2.astype(np.float64))
    bound = {"dW2": dh2.T @ np.abs(fw["h1"]), "dW1": dh1.T @ np.abs(fw["x"]),
             "db2": dh2.sum(axis=0), "db1": dh1.sum(axis=0), "dw3": np.abs(dz) @ np.abs(fw["h2"])}
    for k, m in bound.items():
        # typical entries sit at the operand roundings' size; a ReLU whose
        # input the roundings move across zero changes whole terms, in a few
        # entries only
        r = (np.abs(g16[k] - g64[k]) / np.maximum(m, 1e-300))[m > 0]
        assert np.median(r) <= 2.0 ** -9 and np.percentile(r, 95) <= 2.0 ** -6, k
        assert not np.array_equal(g16[k], g64[k]), k  # the roundings did apply


def test_adagrad_step_closed_form():
    """w = 1, G = 5, g = 2, lr = 0.5, eps = 0: G -> 9, w -> 1 - 0.5 * 2 / 3."""
    w, G = obw.adagrad(np.ones((3, 2)), np.full((3, 2), 5.0), np.array([1]), np.array([[2.0, -4.0]]),
                       lr=0.5, eps=0.0)
    assert np.array_equal(G, [[5, 5], [9, 21], [5, 5]])
    assert np.allclose(w, [[1, 1], [1 - 1 / 3, 1 + 2 / np.sqrt(21)], [1, 1]], rtol=0, atol=1e-15)


def test_backward_hash_rows_skip_unseen_keys():
    """Hash-table features: gradients reach admitted keys only (the zero row an
    unseen key reads is not a parameter), and equal the plain batch's
    gradients of the same rows once the unadmitted rows read zero."""
    plain = synth.generate("tiny", seed=5, B=32, nonzero_bias=True)
    hb = synth.dynamic_emb(plain, capacity=500, seed=5)
    ref = _zero_cold_rows(plain, 500, synth.DYNEMB_FEATURES)
    rng = np.random.default_rng(2)
    dp = rng.standard_normal((hb.B, hb.F * hb.D))
    dd = rng.standard_normal((hb.B, 3 * hb.D))
    g = obw.backward(hb, dp, dd)
    gr = obw.backward(ref, dp, dd)
    for k in ("dW1", "db1", "dW2", "db2", "dw3", "db3", "dq"):
        assert np.array_equal(g[k], gr[k]), k
    for f in range(hb.F):
        rows, grads = g["rows"][f]
        rr, gg = gr["rows"][f]
        if f in synth.DYNEMB_FEATURES:
            assert rows.max() < 500
            keep = rr < 500
            rr, gg = rr[keep], gg[keep]
        assert np.array_equal(rows, rr) and np.array_equal(grads, gg), f
