"""Row-wise sharded EmbeddingBag pooling over data-parallel ranks.

MultiTowerDIN: integrating DynamicEmb, section 5.1: every large table is split
by rows over the N ranks, rank r holding the contiguous block of rows
[r * ceil(rows / N), (r + 1) * ceil(rows / N)); each rank looks up its own
samples (its slice of the global batch), and an all-to-all brings every
looked-up row from its owner. Section 5.2 sizes that exchange by values (one
row per looked-up id), which is the exchange built here:

  1. route: every id of a row-wise table goes to the rank that owns its row,
     as (table, row within the owner's block), in the order the ids appear;
  2. ids all-to-all (counts first, then the ids);
  3. each owner gathers the rows it was asked for from its block, with the
     library's pooling kernel over bags of one value (an exact row copy);
  4. rows all-to-all back to the ranks that asked;
  5. each rank pools its bags from the rows it received, in the bags' own
     value order, with the same pooling kernel over a table made of those rows.

Because step 5 adds a bag's rows in the bag's order, the pooled rows equal
those of unsharded pooling bit for bit. Tables not marked row-wise are held
whole by every rank and pooled locally (data-parallel tables); a table-wise
table is the row-wise case with a single owner.

Routing (bucketing ids by owner, the permutations) is torch tensor plumbing on
the ranks' device; the exchange is torch.distributed (NCCL on GPUs, gloo on
CPU); the row gather and the pooling are the `pool` callable, which is the CUDA
library (`cuda_pool`) in production.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, List, Optional, Sequence

import torch
import torch.distributed as dist

ROW_WISE, TABLE_WISE, REPLICATED = "row_wise", "table_wise", "replicated"
ID_RANGE = 0x01  # the DSF_FLAG_ID_RANGE bit: an id outside its table contributes zero
_TSHIFT = 40     # (table << 40 | row) packs a routed id


@dataclasses.dataclass
class ShardPlan:
    """Which rank owns which rows. rows[f]: rows of table f; kinds[f]: ROW_WISE,
    TABLE_WISE (owner[f] holds it whole) or REPLICATED (every rank does)."""
    rows: List[int]
    world: int
    kinds: List[str]
    owner: List[int]

    @staticmethod
    def make(rows: Sequence[int], world: int, row_wise_min_rows: int = 100_000,
             table_wise: Sequence[int] = ()) -> "ShardPlan":
        """Tables of at least row_wise_min_rows rows are row-wise (the pages'
        large DynamicEmb tables); those listed in table_wise go whole to rank
        f % world; the rest are replicated."""
        kinds, owner = [], []
        for f, n in enumerate(rows):
            if f in table_wise:
                kinds.append(TABLE_WISE)
                owner.append(f % world)
            elif n >= row_wise_min_rows:
                kinds.append(ROW_WISE)
                owner.append(-1)
            else:
                kinds.append(REPLICATED)
                owner.append(-1)
        return ShardPlan([int(n) for n in rows], int(world), kinds, owner)

    def block(self, f: int) -> int:
        """Rows per rank of a row-wise table (the last block may be shorter)."""
        return -(-self.rows[f] // self.world)

    def local_range(self, f: int, rank: int):
        """Rows [lo, hi) of table f that rank holds."""
        k = self.kinds[f]
        if k == REPLICATED:
            return 0, self.rows[f]
        if k == TABLE_WISE:
            return (0, self.rows[f]) if rank == self.owner[f] else (0, 0)
        b = self.block(f)
        return min(rank * b, self.rows[f]), min((rank + 1) * b, self.rows[f])

    def routed(self, f: int) -> bool:
        return self.kinds[f] != REPLICATED

    def owner_of(self, f: int, ids: torch.Tensor) -> torch.Tensor:
        """Owner rank of each id of a routed table; -1 for ids outside it."""
        ok = (ids >= 0) & (ids < self.rows[f])
        if self.kinds[f] == TABLE_WISE:
            own = torch.full_like(ids, self.owner[f])
        else:
            own = torch.div(ids, self.block(f), rounding_mode="floor")
        return torch.where(ok, own, torch.full_like(ids, -1))


def shard_tables(tables: Sequence[torch.Tensor], plan: ShardPlan, rank: int) -> List[torch.Tensor]:
    """The rows of every table that `rank` holds (copies; empty [0, D] where none)."""
    out = []
    for f, t in enumerate(tables):
        lo, hi = plan.local_range(f, rank)
        out.append(t[lo:hi].contiguous().clone())
    return out


PoolFn = Callable[[List[torch.Tensor], torch.Tensor, torch.Tensor, int, Optional[List[int]]],
                  "tuple[torch.Tensor, int]"]


_WS = {}


def cuda_pool(tables: List[torch.Tensor], values: torch.Tensor, lengths: torch.Tensor, B: int,
              pooling: Optional[List[int]] = None):
    """emb_bag_pool of the CUDA library: (pooled [B, F*D] fp32, status bits).
    One workspace per (device, D) is kept and grown to the largest batch seen
    (calls on one device run on its current stream, one after another)."""
    from . import binding
    dev = values.device
    D = int(tables[0].shape[1])
    et = binding.EmbeddingTables([t if t.shape[0] > 0 else t.new_zeros(1, D) for t in tables], pooling)
    key = (str(dev), D)
    ws = _WS.get(key)
    if ws is None or ws.B < B:
        ws = _WS[key] = binding.Workspace(max(B, 1, 2 * (ws.B if ws is not None else 0)), D, device=dev)
    out = torch.empty(B, len(tables) * D, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    binding.emb_bag_pool(et, values, lengths, B, out, ws, status=st)
    return out, binding.read_status(st)


class RowWiseEmbeddingBag:
    """Pooled embeddings of this rank's samples from tables sharded by `plan`.

    local_tables: this rank's rows of every table (shard_tables); pool: the
    pooling primitive (cuda_pool in production); exchange(send, counts) ->
    (received, counts per source): the all-to-all, torch.distributed's
    all_to_all_single over `group` unless given. forward(values, lengths, B)
    takes this rank's KJT (key-major: all values of table 0, then table 1 ...;
    lengths [F * B] int32) and returns (pooled [B, F * D] fp32, status bits).
    Plain (not hash-table) tables, fp32 or bf16; the received rows are fp32
    (exact copies of bf16 rows), so with bf16 tables the replicated ones are
    pooled from fp32 copies kept here."""

    def __init__(self, plan: ShardPlan, local_tables: Sequence[torch.Tensor], rank: int, pool: PoolFn,
                 pooling: Optional[Sequence[int]] = None, group=None, exchange=None):
        self.plan, self.rank, self.pool, self.group = plan, int(rank), pool, group
        self.exchange = exchange if exchange is not None else self._a2a
        self.tables = list(local_tables)
        self.F = len(self.tables)
        self.D = int(self.tables[0].shape[1])
        self.pooling = None if pooling is None else [int(x) for x in pooling]
        self.lo = [plan.local_range(f, rank)[0] for f in range(self.F)]
        self.pool_tables = [t if t.dtype == torch.float32 or plan.routed(f) else t.float().contiguous()
                            for f, t in enumerate(self.tables)]

    def _a2a(self, send: torch.Tensor, counts: List[int]) -> "tuple[torch.Tensor, List[int]]":
        """all-to-all of send (dim 0 split by counts) over torch.distributed;
        returns what arrived and the counts per source rank."""
        W = self.plan.world
        if W == 1:
            return send.clone(), list(counts)
        c = torch.tensor(counts, dtype=torch.int64, device=send.device)
        rc = torch.empty_like(c)
        dist.all_to_all_single(rc, c, group=self.group)
        rcounts = [int(x) for x in rc.tolist()]
        out = send.new_empty((sum(rcounts),) + tuple(send.shape[1:]))
        dist.all_to_all_single(out, send, output_split_sizes=rcounts, input_split_sizes=counts,
                               group=self.group)
        return out, rcounts

    def forward(self, values: torch.Tensor, lengths: torch.Tensor, B: int):
        F, D, plan, dev = self.F, self.D, self.plan, values.device
        lens = lengths.to(torch.int64).clamp_min(0).view(F, B)
        per_f = lens.sum(dim=1)
        starts = torch.cumsum(per_f, 0) - per_f
        n_keys = int(per_f.sum())
        vals = values[:n_keys]
        feat = torch.repeat_interleave(torch.arange(F, device=dev), per_f)
        # 1. route the ids of routed tables: owner, packed (table, local row)
        owner = torch.full_like(vals, -1)
        packed = torch.zeros_like(vals)
        routed = torch.zeros(n_keys, dtype=torch.bool, device=dev)
        for f in range(F):
            if not plan.routed(f):
                continue
            a, n = int(starts[f]), int(per_f[f])
            ids = vals[a:a + n]
            own = plan.owner_of(f, ids)
            lo = torch.div(ids, plan.block(f), rounding_mode="floor") * plan.block(f) \
                if plan.kinds[f] == ROW_WISE else torch.zeros_like(ids)
            owner[a:a + n] = own
            packed[a:a + n] = (f << _TSHIFT) | (ids - lo).clamp_min(0)
            routed[a:a + n] = True
        flags = ID_RANGE if bool((routed & (owner < 0)).any()) else 0
        send_idx = torch.nonzero(routed & (owner >= 0)).squeeze(1)
        order = torch.argsort(owner[send_idx], stable=True)
        send_idx = send_idx[order]
        counts = torch.bincount(owner[send_idx], minlength=plan.world).tolist()
        # 2. ids to their owners
        req, rcounts = self.exchange(packed[send_idx], counts)
        # 3. the owner's row copies: bags of one value over its blocks
        rows_out = self._gather(req)
        # 4. rows back to the ranks that asked
        got, _ = self.exchange(rows_out, rcounts)
        # 5. a table per routed feature made of the rows its values received,
        # in value order (routed ids outside their table keep a zero row)
        recv = torch.zeros(n_keys, D, dtype=torch.float32, device=dev)
        recv[send_idx] = got
        tables, vvals = [], torch.empty_like(vals)
        for f in range(F):
            a, n = int(starts[f]), int(per_f[f])
            if plan.routed(f):
                tables.append(recv[a:a + n].contiguous() if n > 0 else recv.new_zeros(1, D))
                vvals[a:a + n] = torch.arange(n, device=dev)
            else:
                tables.append(self.pool_tables[f])
                vvals[a:a + n] = vals[a:a + n]
        pooled, st = self.pool(tables, vvals, lengths, B, self.pooling)
        return pooled, flags | st

    def _gather(self, req: torch.Tensor) -> torch.Tensor:
        """Rows [n, D] fp32 for the packed requests, in request order."""
        n = int(req.numel())
        out = torch.zeros(n, self.D, dtype=torch.float32, device=req.device)
        if n == 0:
            return out
        tab = torch.div(req, 1 << _TSHIFT, rounding_mode="floor")
        row = req - (tab << _TSHIFT)
        for f in torch.unique(tab).tolist():
            m = torch.nonzero(tab == f).squeeze(1)
            one = torch.ones(int(m.numel()), dtype=torch.int32, device=req.device)
            r, _ = self.pool([self.tables[f]], row[m], one, int(m.numel()), None)
            out[m] = r
        return out
