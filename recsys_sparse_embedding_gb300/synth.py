"""Seeded synthetic inputs for the MultiTowerDIN sparse forward.

This module only draws random numbers in the shapes of the workloads: tables,
KeyedJaggedTensor ids and lengths, sequence ids and lengths, and attention-MLP
weights. It holds none of the method's arithmetic, so the CPU oracle and the
CUDA path can both be fed from it without sharing any computation.

Workload shapes follow the Taobao MultiTowerDIN description ("MultiTowerDIN:
current state analysis", section 1 feature table: 16 deep features, dim 16,
batch 8192, sequence cap 100) and the DynamicEmb follow-up page (section 2.1:
N(0, 0.05) embedding init; section 7: the seq group reads adgroup/cate/brand).
The Taobao ODPS tables themselves are not available; these draws stand in for
them with the same table sizes, batch size, id skew and length mix.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

# Page 1, section 1 feature table, in table order; price is a raw feature with
# 100 boundaries, hence 101 buckets.
TAOBAO_FEATURES = [
    ("user_id", 1_141_730), ("adgroup_id", 846_812), ("campaign_id", 423_438),
    ("brand", 461_498), ("customer", 255_877), ("cate_id", 12_961),
    ("cms_segid", 98), ("cms_group_id", 14), ("final_gender_code", 3),
    ("age_level", 8), ("pvalue_level", 5), ("shopping_level", 5),
    ("occupation", 3), ("new_user_class_level", 6), ("pid", 20), ("price", 101),
]
TAOBAO_ROWS = [n for _, n in TAOBAO_FEATURES]

# Target / sequence sub-feature tables. The literal workload map is {1, 5, 2}
# (adgroup_id, cate_id, campaign_id); the pages' own map is adgroup/cate/brand
# = {1, 5, 3}. Both are arguments of the library; the default is the literal one.
SEQ_TABLES_LITERAL = (1, 5, 2)
SEQ_TABLES_PAGES = (1, 5, 3)

ATTN_N1 = 256   # attn_mlp hidden_units [256, 64]
ATTN_N2 = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    rows: Sequence[int]
    D: int = 16
    dtype: str = "f32"                  # table storage: "f32" or "bf16"
    ids: str = "zipf"                   # "zipf" or "uniform"
    zipf_s: float = 1.1
    multi_hot: Sequence[int] = ()       # features with bag length U{1..8}
    seq_len: str = "geometric"          # "uniform0_10", "geometric", "lognormal", "uniform1_100"
    seq_mean: float = 5.0
    max_len: int = 100
    seq_table: Sequence[int] = SEQ_TABLES_LITERAL

    @property
    def F(self) -> int:
        return len(self.rows)

    @property
    def Q(self) -> int:
        return 3 * self.D

    @property
    def K1(self) -> int:
        return 4 * self.Q


WORKLOADS = {
    "tiny": Workload("tiny", B=64, rows=[1000] * 16, ids="uniform",
                     seq_len="uniform0_10"),
    "taobao": Workload("taobao", B=8192, rows=TAOBAO_ROWS, ids="zipf",
                       zipf_s=1.1, seq_len="geometric", seq_mean=5.0),
    "long_multihot": Workload("long_multihot", B=8192, rows=TAOBAO_ROWS,
                              ids="zipf", zipf_s=1.05,
                              multi_hot=(0, 1, 2, 3, 4), seq_len="lognormal"),
    "gather_stress": Workload(
        "gather_stress", B=65536,
        rows=[2_000_000, 4_000_000, 6_000_000, 8_000_000, 10_000_000] + TAOBAO_ROWS[5:],
        ids="uniform", seq_len="uniform1_100"),
    "wide_bf16": Workload("wide_bf16", B=32768, rows=TAOBAO_ROWS, D=64,
                          dtype="bf16", ids="zipf", zipf_s=1.1,
                          seq_len="geometric", seq_mean=8.0, max_len=200),
}
WORKLOAD_ORDER = ["tiny", "taobao", "long_multihot", "gather_stress", "wide_bf16"]


@dataclasses.dataclass
class Batch:
    """One batch of host inputs (numpy), in the library's layouts.

    tables      list of F arrays [rows_f, D]; float32, or uint16 holding bf16 bits
    lengths     int32 [F*B], key-major (all B bags of feature 0, then feature 1 ...)
    values      int64 [sum(lengths)], the KJT values in the same order
    seq_lengths int32 [B]
    seq_values  int64 [3, P] (P = sum(seq_lengths)), one row per sub-feature
    W1 [N1, K1], b1 [N1], W2 [N2, N1], b2 [N2], w3 [N2], b3 [1]: float32,
    PyTorch Linear layout [out, in].
    """
    wl: Workload
    B: int
    tables: List[np.ndarray]
    lengths: np.ndarray
    values: np.ndarray
    seq_lengths: np.ndarray
    seq_values: np.ndarray
    max_len: int
    q_feat: tuple
    seq_table: tuple
    W1: np.ndarray
    b1: np.ndarray
    W2: np.ndarray
    b2: np.ndarray
    w3: np.ndarray
    b3: np.ndarray
    pooling: Optional[tuple] = None  # per table 0 (sum) / 1 (mean); None: all sum
    # hash-table (DynamicEmb-style) features: f -> int64 keys of the admitted
    # rows, key i owning row i of tables[f]; those features' values (and the
    # sequence values of their sub-features) are raw keys, not row indices
    hash_keys: Optional[dict] = None

    @property
    def F(self) -> int:
        return len(self.tables)

    @property
    def D(self) -> int:
        return self.wl.D

    @property
    def dtype_code(self) -> int:
        return 1 if self.wl.dtype == "bf16" else 0


def _zipf_cdf(n: int, s: float) -> np.ndarray:
    r = np.arange(1, n + 1, dtype=np.float64)
    w = r ** (-s)
    c = np.cumsum(w)
    return c / c[-1]


_CDF_CACHE: dict = {}


def draw_ids(rng: np.random.Generator, n_rows: int, count: int, kind: str,
             s: float) -> np.ndarray:
    """Row ids in [0, n_rows): uniform, or Zipf(s) with rank r -> id r-1
    (hot ids are the low rows) drawn by inverse CDF."""
    if count == 0:
        return np.zeros(0, dtype=np.int64)
    if kind == "uniform" or n_rows == 1:
        return rng.integers(0, n_rows, size=count, dtype=np.int64)
    key = (n_rows, s)
    cdf = _CDF_CACHE.get(key)
    if cdf is None:
        cdf = _zipf_cdf(n_rows, s)
        if len(_CDF_CACHE) > 64:
            _CDF_CACHE.clear()
        _CDF_CACHE[key] = cdf
    u = rng.random(count)
    ids = np.searchsorted(cdf, u, side="right").astype(np.int64)
    return np.minimum(ids, n_rows - 1)


def draw_seq_lengths(rng: np.random.Generator, wl: Workload, B: int) -> np.ndarray:
    if wl.seq_len == "uniform0_10":
        L = rng.integers(0, 11, size=B)
    elif wl.seq_len == "geometric":
        # geometric on {0, 1, ...} with the given mean: p = 1 / (mean + 1)
        L = rng.geometric(1.0 / (wl.seq_mean + 1.0), size=B) - 1
    elif wl.seq_len == "lognormal":
        z = rng.standard_normal(B)
        L = np.rint(np.exp(math.log(30.0) + 0.8 * z))
    elif wl.seq_len == "uniform1_100":
        L = rng.integers(1, 101, size=B)
    else:
        raise ValueError(wl.seq_len)
    return np.minimum(L, wl.max_len).astype(np.int32)


def draw_table(rng: np.random.Generator, rows: int, D: int, dtype: str,
               std: float) -> np.ndarray:
    t = rng.standard_normal((rows, D), dtype=np.float32)
    t *= np.float32(std)
    if dtype == "bf16":
        return f32_to_bf16_bits(t)
    return t


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Draw-time storage conversion of float32 samples to bf16 (torch's
    round-to-nearest-even cast), returned as uint16 bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32)


def xavier_uniform(rng: np.random.Generator, out_f: int, in_f: int,
                   scale: float = 1.0) -> np.ndarray:
    a = math.sqrt(6.0 / (in_f + out_f))
    return (rng.uniform(-a, a, size=(out_f, in_f)) * scale).astype(np.float32)


def generate(wl_name: str, seed: int = 0, B: Optional[int] = None,
             rows: Optional[Sequence[int]] = None, peaked: bool = False,
             nonzero_bias: bool = False,
             seq_table: Optional[Sequence[int]] = None,
             ids_only: bool = False) -> Batch:
    """Draw one batch of the named workload.

    B / rows override the batch size and table sizes (for small parity cases
    that keep the workload's distributions). peaked=True draws tables N(0, 1)
    and scales the MLP weights by 4 so the softmax is far from uniform.
    nonzero_bias=True draws all biases U(-0.1, 0.1) instead of zeros.
    ids_only=True skips drawing the tables (tables = []); every other field is
    what a full draw with the same arguments gives (separate random streams).
    """
    wl = WORKLOADS[wl_name]
    B = wl.B if B is None else int(B)
    rows = list(wl.rows if rows is None else rows)
    st = tuple(wl.seq_table if seq_table is None else seq_table)
    ss = np.random.SeedSequence([seed, WORKLOAD_ORDER.index(wl_name)])
    r_tab, r_ids, r_len, r_seq, r_mlp = [np.random.Generator(np.random.PCG64(s))
                                         for s in ss.spawn(5)]
    F, D = len(rows), wl.D
    std = 1.0 if peaked else 0.05
    tables = [] if ids_only else [draw_table(r_tab, n, D, wl.dtype, std) for n in rows]

    # deep KJT: key-major lengths, then ids per feature
    lengths = np.ones((F, B), dtype=np.int32)
    for f in wl.multi_hot:
        if f < F:
            lengths[f] = r_len.integers(1, 9, size=B)
    vals = [draw_ids(r_ids, rows[f], int(lengths[f].sum()), wl.ids, wl.zipf_s)
            for f in range(F)]
    values = np.concatenate(vals) if vals else np.zeros(0, np.int64)

    seq_lengths = draw_seq_lengths(r_len, wl, B)
    P = int(seq_lengths.sum())
    seq_values = np.stack([draw_ids(r_seq, rows[t], P, wl.ids, wl.zipf_s)
                           for t in st]) if P else np.zeros((3, 0), np.int64)

    scale = 4.0 if peaked else 1.0
    K1 = 4 * 3 * D
    W1 = xavier_uniform(r_mlp, ATTN_N1, K1, scale)
    W2 = xavier_uniform(r_mlp, ATTN_N2, ATTN_N1, scale)
    w3 = xavier_uniform(r_mlp, 1, ATTN_N2, scale).reshape(ATTN_N2)
    if nonzero_bias:
        b1 = r_mlp.uniform(-0.1, 0.1, ATTN_N1).astype(np.float32)
        b2 = r_mlp.uniform(-0.1, 0.1, ATTN_N2).astype(np.float32)
        b3 = r_mlp.uniform(-0.1, 0.1, 1).astype(np.float32)
    else:
        b1 = np.zeros(ATTN_N1, np.float32)
        b2 = np.zeros(ATTN_N2, np.float32)
        b3 = np.zeros(1, np.float32)
    return Batch(wl=wl, B=B, tables=tables, lengths=lengths.reshape(-1),
                 values=values, seq_lengths=seq_lengths,
                 seq_values=np.ascontiguousarray(seq_values, dtype=np.int64),
                 max_len=wl.max_len, q_feat=st, seq_table=st,
                 W1=W1, b1=b1, W2=W2, b2=b2, w3=w3, b3=b3)


def table_bytes(b: Batch) -> int:
    return sum(int(t.nbytes) for t in b.tables)


TOWER_SHAPES = (("Wd1", (512, 256)), ("bd1", (512,)), ("Wd2", (256, 512)), ("bd2", (256,)),
                ("Wd3", (128, 256)), ("bd3", (128,)), ("Wf1", (64, 176)), ("bf1", (64,)),
                ("wo", (64,)), ("bo", (1,)))


def tower_weights(seed: int = 0, bias: float = 0.1) -> list:
    """Random-init dense-tower weights in [out, in] layout, in TOWER_SHAPES
    order: Xavier-uniform matrices (wo as a [1, 64] matrix) and biases drawn
    U(-bias, bias), all float32."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x70A3])))
    out = []
    for name, shape in TOWER_SHAPES:
        if name == "wo":
            out.append(xavier_uniform(rng, 1, shape[0]).reshape(shape))
        elif len(shape) == 2:
            out.append(xavier_uniform(rng, shape[0], shape[1]))
        else:
            out.append(rng.uniform(-bias, bias, shape).astype(np.float32))
    return out


# The five tables above 100K rows that the DynamicEmb migration moves to hash
# tables (user_id, adgroup_id, campaign_id, brand, customer), and its
# per-GPU capacity of 300K rows.
DYNEMB_FEATURES = (0, 1, 2, 3, 4)
DYNEMB_CAPACITY = 300_000
KEY_BITS = 56  # raw keys are drawn from [0, 2^56)


def dynamic_emb(batch: Batch, features: Sequence[int] = DYNEMB_FEATURES,
                capacity: int = DYNEMB_CAPACITY, seed: int = 0) -> Batch:
    """The same batch with `features` served from hash tables.

    Every row r of such a feature's vocabulary gets a distinct random raw key
    in [0, 2^56); the ids become those keys. The table holds the rows whose
    rank is below `capacity` -- the Zipf-hot ids, as a frequency-admitted table
    would -- so the ids of the colder rows are unseen keys. Draws come from
    their own stream, so everything else equals the plain batch.
    """
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0xD1E7])))
    F, B = batch.F, batch.B
    tables = list(batch.tables)
    values = batch.values.copy()
    seq_values = batch.seq_values.copy()
    lengths = batch.lengths.reshape(F, B)
    starts = np.concatenate([[0], np.cumsum(lengths.sum(axis=1))])
    hash_keys = {}
    for f in features:
        n = tables[f].shape[0]
        keys = np.unique(rng.integers(0, 1 << KEY_BITS, size=n + n // 8 + 16, dtype=np.int64))
        keys = rng.permutation(keys)[:n]
        if keys.size < n:
            raise RuntimeError("not enough distinct keys")
        cap = min(capacity, n)
        hash_keys[f] = np.ascontiguousarray(keys[:cap])
        tables[f] = np.ascontiguousarray(tables[f][:cap])
        seg = slice(int(starts[f]), int(starts[f + 1]))
        values[seg] = keys[values[seg]]
        for k, t in enumerate(batch.seq_table):
            if t == f:
                seq_values[k] = keys[seq_values[k]]
    return dataclasses.replace(batch, tables=tables, values=values, seq_values=seq_values,
                               hash_keys=hash_keys)
