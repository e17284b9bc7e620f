"""The parity gate of the backward, as CPU code (numpy): the GPU's
intermediates and gradients against the backward oracle. The GPU tests call
it on device results; tests/test_bwd_gate.py calls it on planted mistakes.

Two evaluations of the backward with the same inputs and the same operand
roundings differ continuously (fp32 sums in another order) except where a
step function lies on the path: a ReLU whose input is within accumulated
rounding error of zero may be taken either way, and a bf16 rounding whose
input is within that error of a rounding boundary may go to the other
neighbour. The oracle bounds, per intermediate, where such events can happen
and how far they can move it (candidates). The gate
  1. checks each GPU intermediate (x, h1, h1 W2^T, dh2, dh2 W2, dh1) against
     the oracle's: equal up to continuous error, and different by more only
     at candidate events, by no more than the candidate bound;
  2. carries the differences actually observed in 1 down to the gradients
     (first-order absolute sums: the slack of each entry);
  3. holds every gradient entry to TOL x (its sum of absolute terms) plus its
     slack, and the entries whose slack is small (unflagged) to TOL x that
     sum alone: the largest ratio there is at most 2^-8 in bf16 mode and
     2^-13 in fp32 mode.
"""
from __future__ import annotations

import numpy as np

from oracle import backward as obw

TOL = {False: 2.0 ** -13, True: 2.0 ** -8}
TOL_MEDIAN = {False: 2.0 ** -16, True: 2.0 ** -12}
FLAG = 1.0 / 8          # flagged: the slack exceeds this fraction of TOL x the magnitude sum
SLACK_FACTOR = 1.25     # first-order slack, with room for second-order terms
REL = 1.0 + 2.0 ** -20  # bounds compared in float64 after fp32 arithmetic


class GateError(AssertionError):
    pass


def _require(ok, msg):
    if not ok:
        raise GateError(msg)


def check_intermediates(ref, v, bf16, b2):
    """v: the GPU's intermediates over the valid positions as float64 arrays
    (keys x, h1, h2 = h1 W2^T, dh2, g = dh2 W2, dh1). Each is held to the
    oracle's value within a bound built from its own accumulation error and
    the differences observed in its inputs; a ReLU may be taken the other way
    only where its input lies within that bound of zero, a bf16 rounding may
    go to the other neighbour only where the bound reaches a rounding
    boundary. Returns the observed differences and masks for observed_slack;
    raises GateError otherwise."""
    it, cd = ref["inter"], ref["cand"]
    U = obw.ACC_UNIT
    x, W2, w3 = it["x"], it["W2"], it["w3"]
    aW2, aw3 = np.abs(W2), np.abs(w3)
    samp, a, da, c, dz = it["samp"], it["a"], it["da"], it["c"], it["dz"]
    B = it["c"].size

    def within(what, d, bound):
        bad = np.abs(d) > bound * REL
        _require(not bad.any(), "%s: %d entries beyond their bound" % (what, int(bad.sum())))
    if bf16:
        _require(np.array_equal(v["x"], x), "x differs from the oracle's bf16 operands")
    else:
        within("x", v["x"] - x, 2.0 ** -24 * np.abs(x))
    # layer 1: h1 = round(ReLU(x W1^T + b1))
    d_h1 = v["h1"] - it["h1"]
    within("h1", d_h1, cd["h1"])
    m1g, m1o = v["h1"] > 0, it["pre1"] > 0
    flip1 = m1g != m1o
    _require(not flip1[~cd["amb1"]].any(), "layer-1 ReLU taken the other way where |pre1| exceeds its bound")
    # layer 2: pre2 = h1 W2^T + b2 (the bias added in fp32)
    pre2g = (v["h2"].astype(np.float32) + np.asarray(b2, np.float32)[None, :]).astype(np.float64)
    b_pre2 = cd["acc2"] + np.abs(d_h1) @ aW2.T + 2.0 ** -24 * np.abs(pre2g)
    within("h1 W2^T + b2", pre2g - it["pre2"], b_pre2)
    m2g, m2o = pre2g > 0, it["pre2"] > 0
    flip2 = m2g != m2o
    _require(not flip2[np.abs(it["pre2"]) > b_pre2 * REL].any(),
             "layer-2 ReLU taken the other way where |pre2| exceeds its bound")
    # softmax and dz, from the observed h2 = ReLU(pre2)
    d_z = np.abs(np.maximum(pre2g, 0) - it["h2"]) @ aw3 + cd["accz"]
    mx = np.zeros(B)
    np.maximum.at(mx, samp, d_z)
    d_a = a * np.expm1(d_z + mx[samp]) + a * (cd["Lb"] + 8) * U
    d_c = np.zeros(B)
    np.add.at(d_c, samp, d_a * np.abs(da) + a * cd["acc_da"] + (cd["Lb"] + 2) * U * a * np.abs(da))
    d_dz = d_a * np.abs(da - c[samp]) + a * (cd["acc_da"] + d_c[samp]) + 4 * U * a * (np.abs(da) + np.abs(c[samp]))
    # dh2 = round(dz w3 [pre2 > 0])
    full2 = np.abs(dz)[:, None] * aw3[None, :]
    e2 = d_dz[:, None] * aw3[None, :] * (m2g | m2o) + full2 * flip2 + U * full2
    d_dh2 = v["dh2"] - it["dh2_op"]
    within("dh2", d_dh2, obw.bf16_spread(it["dh2"], e2) if bf16 else e2)
    # g = dh2 W2, then dh1 = round(g [h1 > 0])
    d_g = v["g"] - it["G"]
    within("dh2 W2", d_g, cd["accG"] + np.abs(d_dh2) @ aW2 + 2.0 ** -24 * np.abs(v["g"]))
    e1 = np.abs(d_g) * (m1g & m1o) + np.maximum(np.abs(it["G"]), np.abs(v["g"])) * flip1
    d_dh1 = v["dh1"] - it["dh1_op"]
    within("dh1", d_dh1, obw.bf16_spread(it["dh1"], e1) if bf16 else e1 + 2.0 ** -24 * np.abs(v["dh1"]))
    return dict(h1=d_h1, m1g=m1g, m1o=m1o, pre2=pre2g, m2g=m2g, m2o=m2o, dh2=d_dh2, g=v["g"], dh1=d_dh1,
                counts=dict(relu1=int(flip1.sum()), relu2=int(flip2.sum()),
                            h1=int((d_h1 != 0).sum()) if bf16 else 0,
                            dh2=int((d_dh2 != 0).sum()) if bf16 else 0,
                            dh1=int((d_dh1 != 0).sum()) if bf16 else 0))


def observed_slack(batch, ref, obs):
    """What the observed intermediate differences can move each gradient by
    (first order): dense {name: array} and rows {table: [n, D]} in the
    oracle's row order."""
    it = ref["inter"]
    B, D = batch.B, batch.D
    Q = 3 * D
    samp, a, da, c, dz = it["samp"], it["a"], it["da"], it["c"], it["dz"]
    x, h1, W1, w3 = it["x"], it["h1"], it["W1"], it["w3"]
    aw3 = np.abs(w3)
    s = it["s32"].astype(np.float64)
    ad_h1, ad_dh2, ad_dh1 = np.abs(obs["h1"]), np.abs(obs["dh2"]), np.abs(obs["dh1"])
    # the softmax moves with h2 = ReLU(pre2)
    d_h2 = np.abs(np.maximum(obs["pre2"], 0) - it["h2"])
    d_z = d_h2 @ aw3
    mx = np.zeros(B)
    np.maximum.at(mx, samp, d_z)
    d_a = a * np.expm1(d_z + mx[samp])
    d_c = np.zeros(B)
    np.add.at(d_c, samp, d_a * np.abs(da))
    d_dz = d_a * np.abs(da - c[samp]) + a * d_c[samp]
    live2 = obs["m2g"] | obs["m2o"]
    dense = dict(
        dW1=ad_dh1.T @ np.abs(x),
        dW2=ad_dh2.T @ np.abs(h1) + np.abs(it["dh2_op"]).T @ ad_h1 + ad_dh2.T @ ad_h1,
        db1=np.abs(obs["g"] * obs["m1g"] - it["G"] * obs["m1o"]).sum(axis=0),
        db2=(np.abs(dz)[:, None] * aw3[None, :] * (obs["m2g"] != obs["m2o"])).sum(axis=0)
        + (d_dz[:, None] * aw3[None, :] * live2).sum(axis=0),
        dw3=np.abs(dz) @ d_h2 + d_dz @ np.abs(it["h2"]),
        db3=np.array([d_dz.sum()]))
    s_dx = ad_dh1 @ np.abs(W1)
    qp = np.abs(it["q32"][samp].astype(np.float64))
    s_dq = np.zeros((B, Q))
    np.add.at(s_dq, samp, s_dx[:, :Q] + s_dx[:, 2 * Q:3 * Q] + s_dx[:, 3 * Q:] * np.abs(s))
    s_ds = d_a[:, None] * np.abs(it["ddin"][samp]) + s_dx[:, Q:2 * Q] + s_dx[:, 2 * Q:3 * Q] + s_dx[:, 3 * Q:] * qp
    g_bag = np.zeros((B, batch.F, D))
    for k, f in enumerate(batch.q_feat):
        g_bag[:, f, :] += s_dq[:, k * D:(k + 1) * D]
    rows = {f: v for f, (_, v) in obw.row_sums(batch, g_bag, s_ds, it["j"]).items()}
    return dense, rows


def gate(err, m, slack, bf16, what):
    """err within TOL x m + slack everywhere, within TOL x m where the slack
    is small; returns (largest ratio err / m over unflagged entries, flagged
    entries, entries, median ratio)."""
    tol = TOL[bf16]
    allowed = tol * m + SLACK_FACTOR * slack
    over = err > allowed
    if over.any():
        i = np.argmax(np.where(over, err - allowed, -np.inf))
        raise GateError("%s: %d entries beyond tol x magnitude + slack (worst: err %.3e, magnitude %.3e, "
                        "slack %.3e)" % (what, int(over.sum()), err.flat[i], m.flat[i], slack.flat[i]))
    flagged = slack > FLAG * tol * m
    un = (m > 0) & ~flagged
    r = err[un] / m[un]
    worst = float(r.max()) if r.size else 0.0
    _require(worst <= tol, "%s: unflagged max ratio %.3e above %.3e" % (what, worst, tol))
    rall = err[m > 0] / m[m > 0]
    med = float(np.median(rall)) if rall.size else 0.0
    _require(med <= TOL_MEDIAN[bf16], "%s: median ratio %.3e above %.3e" % (what, med, TOL_MEDIAN[bf16]))
    return worst, int(flagged.sum()), int(m.size), med


def gate_dense(got, ref, slack, bf16):
    out = {}
    for k in ("dW1", "db1", "dW2", "db2", "dw3", "db3"):
        g = np.asarray(got[k], np.float64).reshape(ref[k].shape)
        out[k] = gate(np.abs(g - ref[k]), ref["bounds"][k], slack[k], bf16, k)
    return out


def gate_rows(got_rows, ref, slack_rows, bf16):
    """got_rows: {table: [n, D]} in the oracle's row order."""
    worst, flagged, total = 0.0, 0, 0
    for f, (_, grads) in ref["rows"].items():
        w, fl, n, _ = gate(np.abs(got_rows[f] - grads), ref["rows_abs"][f], slack_rows[f], bf16, "table %d rows" % f)
        worst, flagged, total = max(worst, w), flagged + fl, total + n
    return worst, flagged, total
