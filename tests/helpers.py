"""Shared test plumbing: run the CUDA path on a synthetic batch and compare
with the oracle. Tolerances follow the path's stated accuracy targets:
pooled sums within 1e-6 relative (here: bit-exact, since both sides sum fp32
rows in bag order), attention output within 1e-5 in the fp32 check mode and
within 2e-2 absolute or 1e-2 relative with the bf16 tensor-core MLP."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from recsys_sparse_embedding_gb300 import binding, synth
from recsys_sparse_embedding_gb300.device_batch import to_device

TOL_F32 = (1e-5, 1e-5)          # abs + rel * |ref|
TOL_BF16 = (2e-2, 1e-2)         # abs OR rel
TOL_BF16_EMUL = 2e-3            # vs the oracle with bf16-rounded MLP operands


class DeviceRun:
    def __init__(self, batch, device="cuda"):
        self.batch = batch
        self.db = to_device(batch, device)
        self.ws = binding.Workspace(batch.B, batch.D, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def fwd(self, mode=binding.DSF_MODE_BF16_TC, which="fused", logits=True):
        db = self.db
        mlp = db.mlp(mode)
        self.ws.prepare(mlp)
        B, Q = db.B, 3 * db.D
        dev = db.values.device
        pooled = torch.full((B, db.F * db.D), float("nan"), device=dev)
        din = torch.full((B, Q), float("nan"), device=dev)
        lg = torch.full((max(1, db.seq_values.shape[-1]),), float("nan"), device=dev) if logits else None
        self.status.zero_()
        if which == "fused":
            binding.din_sparse_fwd(db.tables, db.values, db.lengths, db.seq_values, db.seq_lengths,
                                   db.max_len, db.q_feat, db.seq_table, B, mlp, pooled, din,
                                   self.ws, logits=lg, status=self.status)
        elif which == "pool":
            binding.emb_bag_pool(db.tables, db.values, db.lengths, B, pooled, self.ws,
                                 status=self.status)
        elif which == "attn":
            binding.din_jagged_attn(db.tables, db.values, db.lengths, db.seq_values,
                                    db.seq_lengths, db.max_len, db.q_feat, db.seq_table, B, mlp,
                                    din, self.ws, logits=lg, status=self.status)
        torch.cuda.synchronize()
        return (pooled.cpu().numpy(), din.cpu().numpy(),
                None if lg is None else lg.cpu().numpy(), int(self.status.item()))


def sample_ids(B: int, n: int, seed: int = 0) -> np.ndarray:
    if B <= n:
        return np.arange(B, dtype=np.int32)
    rng = np.random.default_rng(seed)
    edge = np.concatenate([np.arange(32), np.arange(B - 32, B)])
    rest = rng.choice(B, size=n - edge.size, replace=False)
    return np.unique(np.concatenate([edge, rest])).astype(np.int32)


def assert_f32_close(got, ref, name=""):
    err = np.abs(got - ref)
    lim = TOL_F32[0] + TOL_F32[1] * np.abs(ref)
    bad = ~(err <= lim)
    assert not bad.any(), "%s: %d elements beyond fp32 tolerance, max err %.3e" % (
        name, int(bad.sum()), float(np.nanmax(err)))


def assert_bf16_close(got, ref, name=""):
    err = np.abs(got - ref)
    ok = (err <= TOL_BF16[0]) | (err <= TOL_BF16[1] * np.abs(ref))
    assert ok.all(), "%s: %d elements beyond bf16 tolerance, max err %.3e" % (
        name, int((~ok).sum()), float(np.nanmax(err)))


def logits_of(batch, samples, lg_dev):
    """GPU logits [n_seq] -> [n_samples, max_len] aligned with the oracle's."""
    off = np.concatenate([[0], np.cumsum(np.maximum(batch.seq_lengths, 0))])
    out = np.full((samples.size, batch.max_len), -np.inf)
    for i, b in enumerate(samples):
        L = min(max(int(batch.seq_lengths[b]), 0), batch.max_len)
        out[i, :L] = lg_dev[off[b]:off[b] + L]
    return out
