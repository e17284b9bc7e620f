"""CPU oracle for the MultiTowerDIN sparse forward (ctypes front end).

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package. The library under
``recsys_sparse_embedding_gb300`` never imports it and shares no code with it;
the C source ``oracle.c`` is the oracle proper (plain loops, one step per
passage of the pages, each cited there).

Parity status of each oracle function (what pins it, in tests/test_oracle.py):
  oracle_offsets       pinned: closed form (all-ones -> iota), hand-counted cases
  oracle_emb_bag_pool  pinned: single-id bag == table row, integer-valued tables
                       against hand sums, permutation invariance, empty bag == 0
  oracle_attn_mlp      pinned: against numpy matmul (a library GEMM) and a
                       selection-matrix MLP whose logits are known in closed form
  oracle_din           pinned: L=1 -> s0, uniform weights -> mean, padded ==
                       jagged, two-position closed-form softmax (sigmoid), the
                       cat order [q, s, q-s, q*s] via selection MLPs, L=0 -> 0
  oracle_towers        pinned: zero weights -> bias path, identity chain, ReLU
                       after every layer, bf16 mode on representable data
  hash_translate       pinned: a brute-force dict on random keys, unseen -> the
                       zero row, key spaces of different tables kept apart
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

FLAG_ID_RANGE = 1
FLAG_NEG_LENGTH = 2
FLAG_SEQ_TRUNC = 4
FLAG_COUNT = 8


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc, -O2, no
    FP contraction so the results are the same on x86-64 and aarch64)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        L.oracle_offsets.argtypes = [P, i64, P]
        L.oracle_offsets.restype = ctypes.c_int
        L.oracle_emb_bag_pool.argtypes = [i32, i32, i32, P, P, P, i32, P, i64, P, P, i32, P]
        L.oracle_emb_bag_pool.restype = ctypes.c_int
        L.oracle_attn_mlp.argtypes = [P, i64, i32, i32, i32, P, P, P, P, P, P, i32, P]
        L.oracle_attn_mlp.restype = ctypes.c_int
        L.oracle_din.argtypes = ([i32, i32, i32, i32, i32, P, P, P, i32, P, i64, P, P, P,
                                  P, i64, P, i32, P, P, P, P, P, P, i32, i32, P, i32,
                                  P, P, P])
        L.oracle_din.restype = ctypes.c_int
        L.oracle_towers.argtypes = [P, P, i64] + [P] * 10 + [i32, P]
        L.oracle_towers.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


class _Tables:
    """Keeps the table arrays alive and exposes the pointer / row arrays."""

    def __init__(self, tables: Sequence[np.ndarray]):
        self.arrs = [np.ascontiguousarray(t) for t in tables]
        self.ptrs = np.array([_ptr(t) for t in self.arrs], dtype=np.uint64)
        self.rows = np.array([t.shape[0] for t in self.arrs], dtype=np.int64)
        self.D = int(self.arrs[0].shape[1])
        self.dtype = 1 if self.arrs[0].dtype == np.uint16 else 0


def offsets(lengths: np.ndarray):
    lengths = _c(lengths, np.int32)
    out = np.zeros(lengths.size + 1, dtype=np.int64)
    flags = lib().oracle_offsets(_ptr(lengths), lengths.size, _ptr(out))
    return out, flags


def _pooling(pooling, F):
    """int32 [F] pooling modes (0 sum, 1 mean), or None."""
    if pooling is None:
        return None
    a = _c(pooling, np.int32)
    if a.size != F:
        raise ValueError("pooling needs one mode per table")
    return a


def emb_bag_pool(tables, values, lengths, B: int, samples: Optional[Sequence[int]] = None,
                 pooling=None):
    """pooled [n_samples, F*D] float32 (fp32 left-to-right bag sums, or those
    sums over the bag length for mean-pooled tables), flags."""
    T = _Tables(tables)
    F = len(T.arrs)
    pl = _pooling(pooling, F)
    values = _c(values, np.int64)
    lengths = _c(lengths, np.int32)
    samples = _c(np.arange(B) if samples is None else samples, np.int32)
    out = np.zeros((samples.size, F * T.D), dtype=np.float32)
    flags = lib().oracle_emb_bag_pool(F, T.D, T.dtype, _ptr(T.ptrs), _ptr(T.rows),
                                      _ptr(pl) if pl is not None else None, B,
                                      _ptr(values), values.size, _ptr(lengths),
                                      _ptr(samples), samples.size, _ptr(out))
    if flags < 0:
        raise MemoryError("oracle_emb_bag_pool")
    return out, flags


def attn_mlp(x, W1, b1, W2, b2, w3, b3, bf16_mlp: bool = False) -> np.ndarray:
    x = _c(x, np.float64)
    n, K1 = x.shape
    W1, b1, W2, b2 = _c(W1, np.float32), _c(b1, np.float32), _c(W2, np.float32), _c(b2, np.float32)
    w3, b3 = _c(w3, np.float32).reshape(-1), _c(b3, np.float32).reshape(-1)
    N1, N2 = W1.shape[0], W2.shape[0]
    z = np.zeros(n, dtype=np.float64)
    rc = lib().oracle_attn_mlp(_ptr(x), n, K1, N1, N2, _ptr(W1), _ptr(b1), _ptr(W2),
                               _ptr(b2), _ptr(w3), _ptr(b3), int(bf16_mlp), _ptr(z))
    if rc != 0:
        raise MemoryError("oracle_attn_mlp")
    return z


def din(tables, values, lengths, B: int, q_feat, seq_table, seq_values, seq_lengths,
        max_len: int, W1, b1, W2, b2, w3, b3, samples=None, padded: bool = False,
        bf16_mlp: bool = False, want_logits: bool = False, pooling=None):
    """din [n_samples, 3D] float64, flags, (logits, weights) if want_logits."""
    T = _Tables(tables)
    F = len(T.arrs)
    pl = _pooling(pooling, F)
    values = _c(values, np.int64)
    lengths = _c(lengths, np.int32)
    seq_values = _c(seq_values, np.int64).reshape(3, -1)
    n_seq = seq_values.shape[1]
    seq_lengths = _c(seq_lengths, np.int32)
    samples = _c(np.arange(B) if samples is None else samples, np.int32)
    W1, b1, W2, b2 = _c(W1, np.float32), _c(b1, np.float32), _c(W2, np.float32), _c(b2, np.float32)
    w3, b3 = _c(w3, np.float32).reshape(-1), _c(b3, np.float32).reshape(-1)
    qf = _c(q_feat, np.int32)
    st = _c(seq_table, np.int32)
    Q = 3 * T.D
    out = np.zeros((samples.size, Q), dtype=np.float64)
    lg = np.zeros((samples.size, max_len), dtype=np.float64) if want_logits else None
    wt = np.zeros((samples.size, max_len), dtype=np.float64) if want_logits else None
    flags = lib().oracle_din(int(padded), int(bf16_mlp), F, T.D, T.dtype, _ptr(T.ptrs),
                             _ptr(T.rows), _ptr(pl) if pl is not None else None, B,
                             _ptr(values), values.size, _ptr(lengths),
                             _ptr(qf), _ptr(st), _ptr(seq_values), n_seq, _ptr(seq_lengths),
                             max_len, _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2), _ptr(w3),
                             _ptr(b3), W1.shape[0], W2.shape[0], _ptr(samples), samples.size,
                             _ptr(out), _ptr(lg) if lg is not None else None,
                             _ptr(wt) if wt is not None else None)
    if flags < 0:
        raise MemoryError("oracle_din")
    if want_logits:
        return out, flags, lg, wt
    return out, flags


KEY_LIMIT = 1 << 56  # raw keys of hash-table features lie in [0, 2^56)


def hash_translate(keys, raw):
    """The hash-table lookup by its definition (MultiTowerDIN: integrating
    DynamicEmb, sections 1 and 3.2): a raw key admitted to the table reads its
    own row, an unseen key reads the constant zero vector. keys: int64 [n],
    key i owning row i; raw: int64 ids. Returns row indices into the table
    with one zero row appended at index n; a raw id outside [0, 2^56) maps to
    -1, an invalid id (flagged, contributes zero)."""
    keys = np.asarray(keys, dtype=np.int64)
    raw = np.asarray(raw, dtype=np.int64)
    order = np.argsort(keys, kind="stable")
    sk = keys[order]
    pos = np.searchsorted(sk, raw)
    pos_c = np.minimum(pos, max(sk.size - 1, 0))
    hit = (pos < sk.size) & (sk[pos_c] == raw) if sk.size else np.zeros(raw.shape, bool)
    out = np.where(hit, order[pos_c] if sk.size else 0, keys.size).astype(np.int64)
    out[(raw < 0) | (raw >= KEY_LIMIT)] = -1
    return out


def resolve_hashed(batch):
    """(tables, values, seq_values) of a batch with its hash-table features
    turned into plain tables: each such table gains the zero row, and its
    ids become row indices by hash_translate. Batches without hash tables
    come back unchanged."""
    hk = getattr(batch, "hash_keys", None)
    if not hk:
        return batch.tables, batch.values, batch.seq_values
    F, B = len(batch.tables), batch.B
    lengths = np.asarray(batch.lengths, np.int64).reshape(F, B)
    starts = np.concatenate([[0], np.cumsum(np.maximum(lengths, 0).sum(axis=1))])
    tables = list(batch.tables)
    values = np.array(batch.values, dtype=np.int64, copy=True)
    seq_values = np.array(batch.seq_values, dtype=np.int64, copy=True).reshape(3, -1)
    for f, keys in hk.items():
        t = tables[f]
        tables[f] = np.concatenate([t, np.zeros((1, t.shape[1]), t.dtype)])
        a, b = int(starts[f]), min(int(starts[f + 1]), values.size)
        values[a:b] = hash_translate(keys, values[a:b])
        for k, tb in enumerate(batch.seq_table):
            if tb == f:
                seq_values[k] = hash_translate(keys, seq_values[k])
    return tables, values, seq_values


def din_batch(batch, samples=None, padded=False, bf16_mlp=False, want_logits=False, pooling=None):
    """oracle_din on a synth.Batch (pooling: the batch's own modes by default;
    hash-table features resolved by resolve_hashed)."""
    if pooling is None:
        pooling = getattr(batch, "pooling", None)
    tables, values, seq_values = resolve_hashed(batch)
    return din(tables, values, batch.lengths, batch.B, batch.q_feat,
               batch.seq_table, seq_values, batch.seq_lengths, batch.max_len,
               batch.W1, batch.b1, batch.W2, batch.b2, batch.w3, batch.b3,
               samples=samples, padded=padded, bf16_mlp=bf16_mlp, want_logits=want_logits,
               pooling=pooling)


def pool_batch(batch, samples=None, pooling=None):
    if pooling is None:
        pooling = getattr(batch, "pooling", None)
    tables, values, _ = resolve_hashed(batch)
    return emb_bag_pool(tables, values, batch.lengths, batch.B, samples, pooling)


def towers(pooled, din, Wd1, bd1, Wd2, bd2, Wd3, bd3, Wf1, bf1, wo, bo, bf16_mlp: bool = False):
    """The dense towers: pooled [n, 256] (float32), din [n, 48] -> logit [n]
    float64 (see oracle_towers)."""
    pooled = _c(pooled, np.float32).reshape(-1, 256)
    din = _c(din, np.float64).reshape(-1, 48)
    n = pooled.shape[0]
    ws = [_c(a, np.float32).reshape(-1) for a in (Wd1, bd1, Wd2, bd2, Wd3, bd3, Wf1, bf1, wo, bo)]
    sizes = (512 * 256, 512, 256 * 512, 256, 128 * 256, 128, 64 * 176, 64, 64, 1)
    for a, sz in zip(ws, sizes):
        if a.size != sz:
            raise ValueError("tower weight of %d elements, expected %d" % (a.size, sz))
    out = np.zeros(n, dtype=np.float64)
    rc = lib().oracle_towers(_ptr(pooled), _ptr(din), n, *[_ptr(a) for a in ws],
                             int(bf16_mlp), _ptr(out))
    if rc != 0:
        raise MemoryError("oracle_towers")
    return out
