"""The backward of the sparse path and the sparse AdaGrad step on the GPU,
through the C ABI, against the backward oracle.

Both sides take the same inputs: the batch, the oracle's pooled rows and the
upstream gradients. The gate (tests/bwd_gate.py) first holds the device's
per-position intermediates (x, h1, h1 W2^T, dh2, dh2 W2, dh1, read from the
backward's workspace) to the oracle's: equal up to each step's accumulation
error and the differences observed in its inputs, with a ReLU taken the other
way only where its input lies within that bound of zero and a bf16 rounding
to the other neighbour only where the bound reaches a rounding boundary.
Then every weight and row gradient is held to 2^-8 (bf16 mode; 2^-13 in fp32
mode) of its sum of absolute terms, plus, where the observed events reach it,
their first-order effect; the entries those events move by more than an
eighth of the tolerance are counted as flagged, all others must meet the
tolerance alone. The set of touched rows is compared exactly."""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward as obw
from recsys_sparse_embedding_gb300 import binding, synth

import bwd_gate
from helpers import DeviceRun
from test_gpu_parity import F32, TC, _custom_batch

pytestmark = pytest.mark.gpu


class Bwd:
    """One backward of a batch on the device, from the oracle's pooled rows."""

    def __init__(self, batch, mode, seed=0, list_cap=None, with_dpooled=True):
        self.batch, self.mode = batch, mode
        run = DeviceRun(batch)
        self.run, self.db = run, run.db
        db = run.db
        rng = np.random.default_rng(seed)
        B, F, D = batch.B, batch.F, batch.D
        self.dpooled = rng.standard_normal((B, F * D)).astype(np.float32) if with_dpooled else None
        self.ddin = rng.standard_normal((B, 3 * D)).astype(np.float32)
        self.pooled = np.ascontiguousarray(oracle.pool_batch(batch)[0], np.float32)
        n_seq = int(db.seq_values.shape[-1])
        cap = list_cap if list_cap is not None else int(db.values.numel()) + 3 * n_seq
        self.grads = binding.MlpGrads(D)
        self.state = binding.SparseState(db.tables, cap)
        self.ws = binding.BwdWorkspace(B, int(db.values.numel()), n_seq, D)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.pooled_t = torch.from_numpy(self.pooled).cuda()
        self.dp_t = None if self.dpooled is None else torch.from_numpy(self.dpooled).cuda()
        self.dd_t = torch.from_numpy(self.ddin).cuda()

    def backward(self):
        db = self.db
        self.status.zero_()
        binding.din_sparse_bwd(db.tables, db.values, db.lengths, db.seq_values, db.seq_lengths, db.max_len,
                               db.q_feat, db.seq_table, self.batch.B, db.mlp(self.mode), self.pooled_t, self.dp_t,
                               self.dd_t, self.grads, self.state, self.ws, status=self.status)
        return binding.read_status(self.status)

    def oracle(self, bf16):
        return obw.backward(self.batch, self.dpooled, self.ddin, bf16=bf16, pooled=self.pooled)

    def views(self, P, bf16):
        return {k: v.float().cpu().numpy().astype(np.float64) for k, v in self.ws.views(P, bf16).items()}

    def storage_rows(self, f, rows):
        """Storage rows of table f's oracle rows (hash-table tables: the slots
        of their admitted keys)."""
        hk = getattr(self.batch, "hash_keys", None) or {}
        if f not in hk:
            return rows
        ht = self.db.tables.hash
        keys = torch.from_numpy(np.ascontiguousarray(hk[f][rows], np.int64)).cuda()
        return ht.find(f, keys).cpu().numpy()


def check(bw, ref, bf16):
    """The gate on one backward; returns its statistics."""
    P = ref["inter"]["samp"].size
    obs = bwd_gate.check_intermediates(ref, bw.views(P, bf16), bf16, bw.batch.b2)
    dense_s, rows_s = bwd_gate.observed_slack(bw.batch, ref, obs)
    got = {k: bw.grads[k].cpu().numpy() for k in ("dW1", "db1", "dW2", "db2", "dw3", "db3")}
    dense = bwd_gate.gate_dense(got, ref, dense_s, bf16)
    st = bw.state
    F = bw.batch.F
    expect, got_rows = set(), {}
    for f, (rows, _) in ref["rows"].items():
        srow = bw.storage_rows(f, rows)
        sid = next(g for g in range(F) if st.grad[g].data_ptr() == st.grad[f].data_ptr())
        got_rows[f] = st.grad[f][torch.from_numpy(srow).cuda()].cpu().numpy().astype(np.float64)
        expect |= {(sid << 40) | int(r) for r in srow}
    rows = bwd_gate.gate_rows(got_rows, ref, rows_s, bf16)
    n = int(st.count.item())
    listed = set(st.list[:n].cpu().numpy().tolist())
    assert n == len(expect) and listed == expect
    return dense, rows, obs["counts"]


def run_case(batch, modes=(F32, TC), seed=0):
    for mode in modes:
        bw = Bwd(batch, mode, seed)
        assert bw.backward() == 0
        bf16 = mode == TC
        dense, (rw, rf, rn), counts = check(bw, bw.oracle(bf16), bf16)
        print("%s: events %s; dense max unflagged ratio / flagged %s; rows max %.1e, flagged %d of %d" % (
            "bf16" if bf16 else "fp32", counts, {k: "%.1e/%d" % (v[0], v[1]) for k, v in dense.items()}, rw, rf, rn))


@pytest.mark.parametrize("seed", [0, 1])
def test_tiny_backward(seed):
    run_case(synth.generate("tiny", seed=seed, nonzero_bias=True), seed=seed)


def test_backward_small_batches_of_full_workloads():
    run_case(synth.generate("taobao", seed=1, B=1000, nonzero_bias=True), seed=1)
    run_case(synth.generate("long_multihot", seed=1, B=600, nonzero_bias=True), seed=2)


def test_backward_taobao_full_size():
    run_case(synth.generate("taobao", seed=0), modes=(TC,), seed=3)


def test_backward_taobao_many_positions():
    """B = 36,000 (about 180 K valid positions, over 1,400 row tiles): db1's
    partial sums, four rows per 128-position tile, fill a buffer sized by the
    position count, several times the rows of the other column sums."""
    b = synth.generate("taobao", seed=4, B=36000)
    assert int(np.minimum(b.seq_lengths, b.max_len).sum()) > 155_648
    run_case(b, modes=(TC,), seed=21)


def test_backward_mean_pooling_and_long_bags():
    rng = np.random.default_rng(4)
    lens = rng.integers(0, 12, size=(16, 200)).astype(np.int32)
    c = _custom_batch(list(rng.integers(0, 120, size=200)), bags_len=lens, seed=4)
    c.pooling = tuple(1 if f in (1, 3, 5) else 0 for f in range(16))
    run_case(c, seed=4)


def test_backward_edges():
    run_case(_custom_batch([0, 0, 0]), seed=5)            # no positions at all
    run_case(_custom_batch([7]), seed=6)                  # one sample
    run_case(_custom_batch([250, 3, 130, 0], max_len=100), seed=7)   # truncated sequences


def test_backward_hashed_tables():
    b = synth.dynamic_emb(synth.generate("taobao", seed=2, B=800, nonzero_bias=True), seed=2)
    run_case(b, seed=8)
    t = synth.dynamic_emb(synth.generate("tiny", seed=3, nonzero_bias=True), capacity=600, seed=3)
    run_case(t, seed=9)


def test_backward_without_dpooled():
    b = synth.generate("tiny", seed=7, nonzero_bias=True)
    bw = Bwd(b, F32, seed=10, with_dpooled=False)
    assert bw.backward() == 0
    check(bw, bw.oracle(False), False)


def test_list_overflow_is_flagged():
    b = synth.generate("tiny", seed=8, nonzero_bias=True)
    bw = Bwd(b, F32, seed=11, list_cap=10)
    assert bw.backward() & binding.FLAG_GRAD_LIST


def test_adagrad_step_and_state_reset():
    """Two training steps: each backward's row gradients, AdaGrad applied to
    exactly the touched rows (checked against the update formula on the
    kernel's own gradients), and the gradient state zero again afterwards."""
    b = synth.generate("tiny", seed=9, nonzero_bias=True)
    bw = Bwd(b, TC, seed=12)
    st = bw.state
    tabs = bw.db.tables.tables
    lr, eps = 0.05, 1e-10
    for step in range(2):
        assert bw.backward() == 0
        n = int(st.count.item())
        ent = st.list[:n].cpu().numpy()
        sid, rows = ent >> 40, ent & ((1 << 40) - 1)
        before = {}
        for s in np.unique(sid):
            r = rows[sid == s]
            rt = torch.from_numpy(r).cuda()
            before[int(s)] = (r, st.grad[s][rt].cpu().numpy().astype(np.float64),
                              tabs[s][rt].cpu().numpy().astype(np.float64), st.accum[s][rt].cpu().numpy())
        w_all = [t.clone() for t in tabs]
        binding.emb_adagrad_update(bw.db.tables, st, lr=lr, eps=eps)
        torch.cuda.synchronize()
        for s, (r, g, w, G) in before.items():
            w_ref, G_ref = obw.adagrad(w, G, np.arange(r.size), g, lr=lr, eps=eps)
            rt = torch.from_numpy(r).cuda()
            w_new = tabs[s][rt].cpu().numpy().astype(np.float64)
            G_new = st.accum[s][rt].cpu().numpy().astype(np.float64)
            # fp32 against fp64: a few units of the last place of G, and of
            # the weight and its step (about lr on the first step, G starting at 0)
            assert (np.abs(G_new - G_ref) <= 2.0 ** -21 * G_ref).all()
            assert (np.abs(w_new - w_ref) <= 2.0 ** -20 * (np.abs(w) + lr)).all()
            untouched = torch.ones(tabs[s].shape[0], dtype=torch.bool, device="cuda")
            untouched[rt] = False
            assert torch.equal(tabs[s][untouched], w_all[s][untouched])
        assert int(st.count.item()) == 0
        for s in range(len(st.grad)):
            assert not st.grad[s].any() and not st.touched[s].any()
        # the next step's forward reads the updated tables
        pooled, _, _, _ = bw.run.fwd(TC, logits=False)
        bw.pooled = pooled
        bw.pooled_t = torch.from_numpy(pooled).cuda()


def test_backward_wide_bf16_tables():
    """D = 64 with bf16 tables: Q = 192, x of 768, the tensor-core and fp32 modes."""
    run_case(synth.generate("wide_bf16", seed=1, B=256, nonzero_bias=True), seed=13)


def test_adagrad_on_bf16_tables():
    """The update of bf16 tables: fp32 arithmetic, the new weight rounded to
    nearest-even bf16 (within one bf16 unit of the fp64 update)."""
    b = synth.generate("wide_bf16", seed=2, B=128, nonzero_bias=True)
    bw = Bwd(b, TC, seed=14)
    st = bw.state
    tabs = bw.db.tables.tables
    assert bw.backward() == 0
    n = int(st.count.item())
    ent = st.list[:n].cpu().numpy()
    sid, rows = ent >> 40, ent & ((1 << 40) - 1)
    before = {}
    for s in np.unique(sid):
        rt = torch.from_numpy(rows[sid == s]).cuda()
        before[int(s)] = (rt, st.grad[s][rt].cpu().numpy().astype(np.float64),
                          tabs[s][rt].float().cpu().numpy().astype(np.float64), st.accum[s][rt].cpu().numpy())
    lr = 0.05
    binding.emb_adagrad_update(bw.db.tables, st, lr=lr, eps=1e-10)
    torch.cuda.synchronize()
    for s, (rt, g, w, G) in before.items():
        w_ref, _ = obw.adagrad(w, G, np.arange(rt.numel()), g, lr=lr, eps=1e-10)
        w_new = tabs[s][rt].float().cpu().numpy().astype(np.float64)
        # one bf16 unit (2^-7 relative) of the result, plus fp32 rounding of the step
        assert (np.abs(w_new - w_ref) <= 2.0 ** -8 * np.abs(w_ref) + 2.0 ** -20 * (np.abs(w) + lr) + 1e-30).all()
        assert (w_new != w).any()
    assert int(st.count.item()) == 0


def test_backward_captured_in_a_graph_matches_the_eager_call():
    """din_sparse_bwd captured into a CUDA graph (after an eager call, which
    sets up the library's second stream, so that the capture records its
    fork and join) and replayed: the weight gradients equal the eager call's
    bit for bit; the row gradients, summed with atomics, within 2^-20 of
    their magnitude; the touched-row count the same."""
    bw = Bwd(synth.generate("taobao", seed=6, B=2048), TC, seed=6)
    st = bw.state

    def reset():
        for t in st.grad:
            t.zero_()
        for t in st.touched:
            t.zero_()
        st.count.zero_()

    assert bw.backward() == 0
    dense0 = {k: bw.grads[k].clone() for k in ("dW1", "db1", "dW2", "db2", "dw3", "db3")}
    rows0 = [t.clone() for t in st.grad]
    count0 = int(st.count.item())
    db = bw.db
    reset()
    for k in dense0:
        bw.grads[k].fill_(float("nan"))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.din_sparse_bwd(db.tables, db.values, db.lengths, db.seq_values, db.seq_lengths, db.max_len,
                               db.q_feat, db.seq_table, bw.batch.B, db.mlp(TC), bw.pooled_t, bw.dp_t, bw.dd_t,
                               bw.grads, st, bw.ws, status=bw.status)
    for _ in range(2):
        reset()
        bw.status.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(bw.status.item()) == 0
        for k, v in dense0.items():
            assert torch.equal(bw.grads[k], v), k
        for a, b in zip(st.grad, rows0):
            assert torch.allclose(a, b, rtol=2.0 ** -20, atol=2.0 ** -20 * float(b.abs().max()) + 1e-30)
        assert int(st.count.item()) == count0
