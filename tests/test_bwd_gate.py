"""The backward parity gate on the CPU: the oracle against itself passes;
evaluations that take a ReLU or a bf16 rounding the other way at a candidate
event pass; planted mistakes fail (a doubled row contribution, a position
dropped from a weight gradient, a ReLU or a rounding taken the other way
where the bounds do not allow it)."""
import numpy as np
import pytest

from oracle import backward as obw
from recsys_sparse_embedding_gb300 import synth

import bwd_gate


def _inputs(batch, seed):
    rng = np.random.default_rng(seed)
    dp = rng.standard_normal((batch.B, batch.F * batch.D)).astype(np.float32)
    dd = rng.standard_normal((batch.B, 3 * batch.D)).astype(np.float32)
    return dp, dd


def _views(ref):
    """The intermediates a device run would leave, taken from an oracle run."""
    it = ref["inter"]
    return dict(x=it["x"], h1=it["h1"], h2=it["pre2"] - it["b2"][None, :], dh2=it["dh2_op"], g=it["G"],
                dh1=it["dh1_op"])


def _run_gate(batch, ref, res, bf16):
    """Gate `res` (an oracle result standing for a device result) against ref."""
    obs = bwd_gate.check_intermediates(ref, _views(res), bf16, batch.b2)
    dense_s, rows_s = bwd_gate.observed_slack(batch, ref, obs)
    bwd_gate.gate_dense(res, ref, dense_s, bf16)
    got_rows = {f: res["rows"][f][1] for f in ref["rows"]}
    return bwd_gate.gate_rows(got_rows, ref, rows_s, bf16), obs["counts"]


@pytest.fixture(scope="module", params=[False, True], ids=["fp32", "bf16"])
def case(request):
    b = synth.generate("taobao", seed=3, B=300, nonzero_bias=True)
    dp, dd = _inputs(b, 3)
    return b, dp, dd, request.param, obw.backward(b, dp, dd, bf16=request.param)


def test_oracle_against_itself(case):
    b, dp, dd, bf16, ref = case
    (worst, flagged, total), counts = _run_gate(b, ref, ref, bf16)
    assert worst == 0.0 and flagged == 0 and total > 0
    assert not any(counts.values())


def _flipped_relu1(monkeypatch, batch, dp, dd, bf16, pick):
    """The oracle run with the layer-1 ReLU of one (position, unit) taken the
    other way (its pre-activation negated, h1 following)."""
    orig = obw.forward

    def fwd(*a, **k):
        fw = orig(*a, **k)
        p, u = pick(fw)
        fw["pre1"][p, u] = -fw["pre1"][p, u]
        v = max(fw["pre1"][p, u], 0.0)
        fw["h1"][p, u] = obw.round_bf16(np.array([v]))[0] if bf16 else v
        return fw
    monkeypatch.setattr(obw, "forward", fwd)
    try:
        return obw.backward(batch, dp, dd, bf16=bf16)
    finally:
        monkeypatch.setattr(obw, "forward", orig)


def test_relu_taken_the_other_way_at_a_candidate_passes(case, monkeypatch):
    b, dp, dd, bf16, ref = case
    amb = ref["cand"]["amb1"] & (ref["inter"]["pre1"] != 0)
    assert amb.any()
    p, u = np.argwhere(amb)[0]
    res = _flipped_relu1(monkeypatch, b, dp, dd, bf16, lambda fw: (p, u))
    assert not np.array_equal(res["dW1"], ref["dW1"])
    _, counts = _run_gate(b, ref, res, bf16)
    assert counts["relu1"] == 1


def test_relu_taken_the_other_way_elsewhere_fails(case, monkeypatch):
    b, dp, dd, bf16, ref = case
    pre1 = ref["inter"]["pre1"]
    far = ~ref["cand"]["amb1"] & (np.abs(pre1) > 0)
    p, u = np.argwhere(far)[np.argmin(np.abs(pre1[far]))]   # the nearest to zero outside the candidates
    res = _flipped_relu1(monkeypatch, b, dp, dd, bf16, lambda fw: (p, u))
    with pytest.raises(bwd_gate.GateError, match="ReLU|h1"):
        _run_gate(b, ref, res, bf16)


def test_rounding_to_the_other_neighbour_outside_candidates_fails(case):
    b, dp, dd, bf16, ref = case
    if not bf16:
        pytest.skip("no operand rounding in fp32 mode")
    res = dict(ref, inter=dict(ref["inter"]))
    dh1 = ref["inter"]["dh1_op"].copy()
    p, u = np.argwhere(dh1 != 0)[0]
    dh1[p, u] = obw.round_bf16(np.array([dh1[p, u] * (1 + 2.0 ** -7)]))[0]   # the next bf16 value up
    assert dh1[p, u] != ref["inter"]["dh1_op"][p, u]
    res["inter"]["dh1_op"] = dh1
    with pytest.raises(bwd_gate.GateError, match="dh1"):
        _run_gate(b, ref, res, bf16)


def _row_counts(batch, ref):
    ones_bag = np.ones((batch.B, batch.F, batch.D))
    ones_pos = np.ones((ref["inter"]["samp"].size, 3 * batch.D))
    return {f: v[:, 0] for f, (_, v) in obw.row_sums(batch, ones_bag, ones_pos, ref["inter"]["j"]).items()}


def test_doubled_bag_contribution_fails(case):
    """One value of one bag adds its bag's gradient to its row twice."""
    b, dp, dd, bf16, ref = case
    counts = _row_counts(b, ref)
    f = next(f for f in range(b.F) if f not in b.q_feat and f not in b.seq_table)
    rows, grads = ref["rows"][f]
    lengths = np.asarray(b.lengths).reshape(b.F, b.B)
    start = int(lengths[:f].sum())
    bag = np.repeat(np.arange(b.B), lengths[f])
    vals = np.asarray(b.values[start:start + int(lengths[f].sum())])
    i = next(i for i, v in enumerate(vals) if counts[f][np.searchsorted(rows, v)] == 1)
    k = np.searchsorted(rows, vals[i])
    planted = grads.copy()
    planted[k] += dp[bag[i], f * b.D:(f + 1) * b.D]
    got = {g: (planted if g == f else ref["rows"][g][1]) for g in ref["rows"]}
    zero = {g: np.zeros_like(v) for g, v in ref["rows_abs"].items()}
    bwd_gate.gate_rows({g: ref["rows"][g][1] for g in ref["rows"]}, ref, zero, bf16)
    with pytest.raises(bwd_gate.GateError, match="table %d rows" % f):
        bwd_gate.gate_rows(got, ref, zero, bf16)


def test_doubled_sequence_contribution_fails(case):
    """One position's sequence-row gradient is added to its row twice."""
    b, dp, dd, bf16, ref = case
    counts = _row_counts(b, ref)
    it = ref["inter"]
    D = b.D
    seq = np.asarray(b.seq_values).reshape(3, -1)
    for p in range(it["samp"].size):
        tb = b.seq_table[0]
        rid = seq[0, it["j"][p]]
        rows, grads = ref["rows"][tb]
        k = np.searchsorted(rows, rid)
        if k < rows.size and rows[k] == rid and counts[tb][k] == 1:
            break
    planted = grads.copy()
    planted[k] += ref["ds"][p, :D]
    got = {g: (planted if g == tb else ref["rows"][g][1]) for g in ref["rows"]}
    zero = {g: np.zeros_like(v) for g, v in ref["rows_abs"].items()}
    with pytest.raises(bwd_gate.GateError, match="table %d rows" % tb):
        bwd_gate.gate_rows(got, ref, zero, bf16)


def test_dropped_position_in_dW1_fails():
    b = synth.generate("taobao", seed=5, B=24, nonzero_bias=True)
    dp, dd = _inputs(b, 5)
    for bf16 in (False, True):
        ref = obw.backward(b, dp, dd, bf16=bf16)
        it = ref["inter"]
        p = int(np.argmax(np.abs(it["dh1_op"]).sum(axis=1)))
        res = dict(ref, dW1=ref["dW1"] - np.outer(it["dh1_op"][p], it["x"][p]))
        zero = {k: np.zeros_like(v) for k, v in ref["bounds"].items()}
        with pytest.raises(bwd_gate.GateError, match="dW1"):
            bwd_gate.gate_dense(res, ref, zero, bf16)
