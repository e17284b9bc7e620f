"""CPU oracle for the backward of the MultiTowerDIN sparse forward and its
sparse AdaGrad step (numpy, float64).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the library.

What it computes, from the forward's definition (MultiTowerDIN: current state
analysis, sections 4.2 and 4.4; the optimizer of section 1: sparse AdaGrad,
lr 1e-3), given the upstream gradients dpooled [B, F*D] and ddin [B, 3D]:
  forward  q_b = pooled query slices, s_t = sequence rows,
           x_t = [q, s_t, q - s_t, q * s_t], h1 = ReLU(W1 x + b1),
           h2 = ReLU(W2 h1 + b2), z_t = w3 . h2 + b3, a = softmax_t(z),
           din_b = sum_t a_t s_t
  backward da_t = ddin . s_t;  dz_t = a_t (da_t - sum_u a_u da_u)
           ds_t = a_t ddin (+ the x path below)
           dh2 = dz w3 * [W2 h1 + b2 > 0];  dw3 += dz h2;  db3 += dz;  db2 += dh2
           dh1 = (W2^T dh2) * [W1 x + b1 > 0];  dW2 += dh2 h1^T;  db1 += dh1
           dx = W1^T dh1;  dW1 += dh1 x^T
           dq += dx_q + dx_d + dx_p * s_t;  ds_t += dx_s - dx_d + dx_p * q
  rows     every value of bag (f, b) receives dpooled[b, f] plus dq_b's slice
           when f is a query feature (over the bag length when f pools by
           mean); row seq_values[k][j] of table seq_table[k] receives the k-th
           slice of ds_t; contributions to one row are summed
  AdaGrad  per touched row: G += g^2 (elementwise); w -= lr g / (sqrt(G) + eps)
bf16=True rounds the GEMM operands to bf16 where the tensor-core path does:
x, W1, W2, h1 (forward, as the forward oracle), dh2 and dh1 (backward).

Pinned in tests/test_oracle.py by central finite differences of the forward
(the oracle's own fp64 forward, itself checked against oracle_din), by an
AdaGrad step in closed form, and by duplicate-row accumulation.
"""
from __future__ import annotations

import numpy as np

from . import pool_batch, resolve_hashed


def round_bf16(a) -> np.ndarray:
    """float32 -> nearest bf16 (ties to even), returned as float64."""
    f = np.asarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    nan = np.isnan(f)
    out = r.astype(np.uint32).view(np.float32).astype(np.float64)
    out[nan] = np.nan
    return out


def _positions(batch):
    """(sample of each valid position, value index j of each position), in
    sample order: positions t < min(L_b, max_len) at j = seq_off[b] + t."""
    L = np.maximum(np.asarray(batch.seq_lengths, np.int64), 0)
    off = np.concatenate([[0], np.cumsum(L)])
    Lc = np.minimum(L, batch.max_len)
    samp = np.repeat(np.arange(batch.B), Lc)
    t = np.arange(int(Lc.sum())) - np.repeat(np.concatenate([[0], np.cumsum(Lc)])[:-1], Lc)
    return samp, off[samp] + t, Lc


def pooled64(batch):
    """Bag sums (or means) in float64, in bag order: the pooled rows when the
    tables are float64 (for finite differences)."""
    tables, values, _ = resolve_hashed(batch)
    F, B, D = batch.F, batch.B, batch.D
    lengths = np.maximum(np.asarray(batch.lengths, np.int64).reshape(F, B), 0)
    off = np.concatenate([[0], np.cumsum(lengths.reshape(-1))])
    pooling = getattr(batch, "pooling", None)
    out = np.zeros((B, F * D))
    for f in range(F):
        for b in range(B):
            acc = np.zeros(D)
            for i in range(int(off[f * B + b]), int(off[f * B + b + 1])):
                v = values[i]
                if 0 <= v < tables[f].shape[0]:
                    acc = acc + tables[f][v]
            if pooling is not None and pooling[f] == 1 and lengths[f, b] > 0:
                acc = acc / lengths[f, b]
            out[b, f * D:(f + 1) * D] = acc
    return out


def forward(batch, bf16=False, pooled=None):
    """The forward quantities the backward needs (float64): q [B, 3D], per
    position s, x, the two pre-activations, h1 as layer 2 reads it, h2, z, the
    softmax weights a and din [B, 3D]. The query and rows keep the tables'
    precision: float32 tables give the fp32 pooled rows of the forward (the C
    oracle's), float64 tables stay float64."""
    D, B = batch.D, batch.B
    Q = 3 * D
    tables, _, seq_values = resolve_hashed(batch)
    wdt = np.float64 if np.asarray(tables[0]).dtype == np.float64 else np.float32
    if pooled is None:
        pooled = pooled64(batch) if wdt == np.float64 else pool_batch(batch)[0]
    pooled = np.asarray(pooled, wdt)
    q32 = np.concatenate([pooled[:, f * D:(f + 1) * D] for f in batch.q_feat], axis=1)
    samp, j, Lc = _positions(batch)
    P = samp.size
    s32 = np.zeros((P, Q), wdt)
    for k, tb in enumerate(batch.seq_table):
        ids = seq_values[k, j] if P else np.zeros(0, np.int64)
        ok = (ids >= 0) & (ids < tables[tb].shape[0])
        rows = np.asarray(tables[tb])
        if rows.dtype == np.uint16:  # bf16 bits
            rows = (rows.astype(np.uint32) << 16).view(np.float32)
        s32[ok, k * D:(k + 1) * D] = rows[ids[ok]]
    qp = q32[samp]
    if bf16:
        x = np.concatenate([round_bf16(qp), round_bf16(s32), round_bf16(qp - s32), round_bf16(qp * s32)], axis=1)
        W1 = round_bf16(batch.W1)
        W2 = round_bf16(batch.W2)
    else:
        q64, s64 = qp.astype(np.float64), s32.astype(np.float64)
        x = np.concatenate([q64, s64, q64 - s64, q64 * s64], axis=1)
        W1 = batch.W1.astype(np.float64)
        W2 = batch.W2.astype(np.float64)
    b1 = batch.b1.astype(np.float64)
    b2 = batch.b2.astype(np.float64)
    w3 = batch.w3.astype(np.float64).reshape(-1)
    b3 = float(np.asarray(batch.b3).reshape(-1)[0])
    acc1 = x @ W1.T
    if bf16:
        pre1 = (acc1.astype(np.float32) + batch.b1.astype(np.float32)).astype(np.float64)
        h1 = round_bf16(np.maximum(pre1, 0.0))
    else:
        pre1 = acc1 + b1
        h1 = np.maximum(pre1, 0.0)
    pre2 = h1 @ W2.T + b2
    h2 = np.maximum(pre2, 0.0)
    z = h2 @ w3 + b3
    # softmax over each sample's valid positions
    a = np.zeros(P)
    din = np.zeros((B, Q))
    starts = np.concatenate([[0], np.cumsum(Lc)])
    for b in np.nonzero(Lc)[0]:
        sl = slice(int(starts[b]), int(starts[b + 1]))
        e = np.exp(z[sl] - z[sl].max())
        a[sl] = e / e.sum()
        din[b] = a[sl] @ s32[sl].astype(np.float64)
    return dict(q32=q32, s32=s32, samp=samp, j=j, Lc=Lc, starts=starts, x=x, W1=W1, W2=W2,
                b1=b1, b2=b2, b3=b3, pre1=pre1, h1=h1, pre2=pre2, h2=h2, z=z, a=a, din=din, w3=w3)


# Per-term relative error allowed for an fp32 sum evaluated in another order:
# twice the unit roundoff of round-to-nearest fp32, so that adders which
# truncate (tensor-core accumulation) are covered as well.
ACC_UNIT = 2.0 ** -22


def bf16_spread(v, e):
    """Largest |bf16(w) - bf16(v)| over |w - v| <= e: rounding to bf16 is
    monotone, so the extremes sit at the two ends of the interval (w is an
    fp32 value, and rounding the ends to fp32 only widens the bound)."""
    r = round_bf16(v)
    return np.maximum(np.abs(round_bf16(v + e) - r), np.abs(round_bf16(v - e) - r))


def error_bounds(fw, bf16, ddin, dh2_op):
    """Where another evaluation of this backward may differ from this one.

    Two evaluations with the same inputs and the same operand roundings
    differ continuously (fp32 sums in another order) except where a step
    function lies on the path: a ReLU whose input is within the accumulated
    rounding error of zero may be taken either way, and a bf16 rounding whose
    input is within that error of a rounding boundary may go to the other
    neighbour. Returns, per quantity, the bound on the rounding error of the
    step that forms it from its inputs (ACC_UNIT per term of its sums):
    C1 and amb1 (|pre1| <= C1: the layer-1 ReLU may go either way), h1 (the
    largest change of bf16(ReLU(pre1)) when pre1 moves by C1), acc2 (of
    h1 W2^T + b2), accz (of w3 . h2 + b3), acc_da (of ddin . s), accG (of
    dh2 W2), Lb (each position's sample length, for the softmax sums)."""
    U = ACC_UNIT
    x, W1, W2, w3 = fw["x"], fw["W1"], fw["W2"], fw["w3"]
    pre1, h1, samp = fw["pre1"], fw["h1"], fw["samp"]
    C1 = (x.shape[1] + 2) * U * (np.abs(x) @ np.abs(W1).T + np.abs(fw["b1"]))
    if bf16:   # h1 = bf16(ReLU(pre1)) is monotone in pre1: its extremes at the ends
        h1b = np.maximum(np.abs(round_bf16(np.maximum(pre1 + C1, 0)) - h1),
                         np.abs(round_bf16(np.maximum(pre1 - C1, 0)) - h1))
    else:
        h1b = C1 * (pre1 > -C1)
    s = fw["s32"].astype(np.float64)
    B = ddin.shape[0]
    Lb = np.bincount(samp, minlength=B)[samp] if samp.size else np.zeros(0)
    return dict(C1=C1, amb1=np.abs(pre1) <= C1, h1=h1b, Lb=Lb,
                acc2=(h1.shape[1] + 2) * U * (np.abs(h1) @ np.abs(W2).T + np.abs(fw["b2"])),
                accz=(w3.size + 2) * U * (np.abs(fw["h2"]) @ np.abs(w3) + abs(fw["b3"])),
                acc_da=(s.shape[1] + 1) * U * np.einsum("pd,pd->p", np.abs(ddin[samp]), np.abs(s)),
                accG=(W2.shape[0] + 1) * U * (np.abs(dh2_op) @ np.abs(W2)))


def backward(batch, dpooled, ddin, bf16=False, pooled=None):
    """Gradients of sum(dpooled * pooled) + sum(ddin * din).

    Returns dict: dW1 [256, 12D], db1, dW2 [64, 256], db2, dw3 [64], db3 [1],
    dq [B, 3D], ds [P, 3D], and rows: {f: (row indices, grads [n, D])} per
    table -- the summed gradient of every row the batch touched (rows of
    hash-table features index their admitted keys; unseen keys, whose zero
    row is not a parameter, and invalid ids get none); rows_abs and bounds:
    each row gradient's and weight gradient's sum of absolute terms, carried
    through the whole chain (|da| = |ddin|.|s|, |dz| = a (|da| + sum a |da|),
    ...), which bounds the rounding errors of any evaluation order; cand: the
    error bounds of error_bounds; inter: the forward and backward
    intermediates (per position: x, pre1, h1, pre2, h2, a, dz, dh2 and its
    operand dh2_op, G = dh2_op W2, dh1 and dh1_op)."""
    fw = forward(batch, bf16, pooled)
    D, B, F = batch.D, batch.B, batch.F
    Q = 3 * D
    ddin = np.asarray(ddin, np.float64).reshape(B, Q)
    dpooled = np.zeros((B, F * D)) if dpooled is None else np.asarray(dpooled, np.float64).reshape(B, F * D)
    samp, a, s = fw["samp"], fw["a"], fw["s32"].astype(np.float64)
    P = samp.size
    # softmax and weighted sum
    da = np.einsum("pd,pd->p", ddin[samp], s)
    c = np.zeros(B)
    np.add.at(c, samp, a * da)
    dz = a * (da - c[samp])
    ds = a[:, None] * ddin[samp]
    # score layer and the two hidden layers
    dh2 = dz[:, None] * fw["w3"][None, :] * (fw["pre2"] > 0)
    dw3 = dz @ fw["h2"]
    db3 = np.array([dz.sum()])
    db2 = dh2.sum(axis=0)
    dh2_op = round_bf16(dh2) if bf16 else dh2
    dW2 = dh2_op.T @ fw["h1"]
    G = dh2_op @ fw["W2"]
    dh1 = G * (fw["pre1"] > 0)
    db1 = dh1.sum(axis=0)
    dh1_op = round_bf16(dh1) if bf16 else dh1
    dW1 = dh1_op.T @ fw["x"]
    dx = dh1_op @ fw["W1"]
    # x = [q, s, q - s, q * s]
    qp = fw["q32"][samp].astype(np.float64)
    dxq, dxs, dxd, dxp = dx[:, :Q], dx[:, Q:2 * Q], dx[:, 2 * Q:3 * Q], dx[:, 3 * Q:]
    dq = np.zeros((B, Q))
    np.add.at(dq, samp, dxq + dxd + dxp * s)
    ds = ds + dxs - dxd + dxp * qp
    # first-order magnitudes: each quantity's sum of absolute terms, through
    # the same chain (rounding errors are bounded by multiples of these)
    da_m = np.einsum("pd,pd->p", np.abs(ddin[samp]), np.abs(s))
    c_m = np.zeros(B)
    np.add.at(c_m, samp, a * da_m)
    dz_m = a * (da_m + c_m[samp])
    dh2_m = dz_m[:, None] * np.abs(fw["w3"])[None, :] * (fw["pre2"] > 0)
    dh1_m = (dh2_m @ np.abs(fw["W2"])) * (fw["pre1"] > 0)
    dx_m = dh1_m @ np.abs(fw["W1"])
    aq = np.abs(qp)
    dq_m = np.zeros((B, Q))
    np.add.at(dq_m, samp, dx_m[:, :Q] + dx_m[:, 2 * Q:3 * Q] + dx_m[:, 3 * Q:] * np.abs(s))
    ds_m = a[:, None] * np.abs(ddin[samp]) + dx_m[:, Q:2 * Q] + dx_m[:, 2 * Q:3 * Q] + dx_m[:, 3 * Q:] * aq
    # row gradients and their magnitude sums
    g_bag = dpooled.reshape(B, F, D).copy()
    g_bag_m = np.abs(g_bag)
    for k, f in enumerate(batch.q_feat):
        g_bag[:, f, :] += dq[:, k * D:(k + 1) * D]
        g_bag_m[:, f, :] += dq_m[:, k * D:(k + 1) * D]
    rows = row_sums(batch, g_bag, ds, fw["j"])
    rows_abs = {f: v for f, (_, v) in row_sums(batch, g_bag_m, ds_m, fw["j"]).items()}
    bounds = dict(dW2=dh2_m.T @ np.abs(fw["h1"]), dW1=dh1_m.T @ np.abs(fw["x"]), db2=dh2_m.sum(axis=0),
                  db1=dh1_m.sum(axis=0), dw3=dz_m @ np.abs(fw["h2"]), db3=np.array([dz_m.sum()]))
    inter = dict(fw, dz=dz, da=da, c=c, dh2=dh2, dh2_op=dh2_op, G=G, dh1=dh1, dh1_op=dh1_op, ddin=ddin)
    return dict(dW1=dW1, db1=db1, dW2=dW2, db2=db2, dw3=dw3, db3=db3, dq=dq, ds=ds, rows=rows,
                rows_abs=rows_abs, bounds=bounds, cand=error_bounds(fw, bf16, ddin, dh2_op), inter=inter,
                din=fw["din"])


def row_sums(batch, g_bag, g_pos, j):
    """Sums per touched row, as the row gradients are formed: every value of
    bag (f, b) receives g_bag[b, f] (divided by the bag length when f pools by
    mean), and row seq_values[k][j_t] of table seq_table[k] receives the k-th
    D-slice of g_pos[t]; ids outside the table, unseen hash keys (the zero
    row) and nothing else are left out. Returns {f: (rows, sums [n, D])}."""
    F, B, D = batch.F, batch.B, batch.D
    tables, values, seq_values = resolve_hashed(batch)
    hk = getattr(batch, "hash_keys", None) or {}
    lengths = np.maximum(np.asarray(batch.lengths, np.int64).reshape(F, B), 0)
    bag_off = np.concatenate([[0], np.cumsum(lengths.reshape(-1))])
    pooling = getattr(batch, "pooling", None)

    def valid(f, ids):
        n = tables[f].shape[0] - (1 if f in hk else 0)   # the zero row is not a parameter
        return (ids >= 0) & (ids < n)
    cf, cr, cg = [], [], []
    for f in range(F):
        lf = lengths[f]
        n = int(lf.sum())
        if n == 0:
            continue
        start = int(bag_off[f * B])
        ids = values[start:start + n]
        bag = np.repeat(np.arange(B), lf)
        g = g_bag[bag, f, :]
        if pooling is not None and pooling[f] == 1:
            g = g / lf[bag][:, None]
        ok = valid(f, ids)
        cf.append(np.full(int(ok.sum()), f)); cr.append(ids[ok]); cg.append(g[ok])
    for k, tb in enumerate(batch.seq_table):
        ids = seq_values[k, j] if j.size else np.zeros(0, np.int64)
        ok = valid(tb, ids)
        cf.append(np.full(int(ok.sum()), tb)); cr.append(ids[ok]); cg.append(g_pos[ok, k * D:(k + 1) * D])
    cf = np.concatenate(cf) if cf else np.zeros(0, np.int64)
    cr = np.concatenate(cr) if cr else np.zeros(0, np.int64)
    cg = np.concatenate(cg) if cg else np.zeros((0, D))
    out = {}
    for f in np.unique(cf):
        m = cf == f
        u, inv = np.unique(cr[m], return_inverse=True)
        acc = np.zeros((u.size, D))
        np.add.at(acc, inv, cg[m])
        out[int(f)] = (u, acc)
    return out


def adagrad(table, accum, rows, grads, lr=1e-3, eps=1e-10):
    """Sparse AdaGrad on the listed rows (float64 copies of the float32 state):
    G += g * g, w -= lr * g / (sqrt(G) + eps); other rows unchanged."""
    w = np.array(table, dtype=np.float64, copy=True)
    G = np.array(accum, dtype=np.float64, copy=True)
    G[rows] += grads * grads
    w[rows] -= lr * grads / (np.sqrt(G[rows]) + eps)
    return w, G
