"""Moves a host batch (numpy arrays from ``synth``) to device tensors in the
library's layouts. Plumbing only: copies, no arithmetic of the method."""
from __future__ import annotations

import dataclasses
from typing import List

import numpy as np
import torch

from . import binding


@dataclasses.dataclass
class DeviceBatch:
    B: int
    D: int
    max_len: int
    q_feat: tuple
    seq_table: tuple
    tables: binding.EmbeddingTables
    values: torch.Tensor       # int64 [n_values]
    lengths: torch.Tensor      # int32 [F*B]
    seq_values: torch.Tensor   # int64 [3, P]
    seq_lengths: torch.Tensor  # int32 [B]
    mlp_t: List[torch.Tensor]  # W1, b1, W2, b2, w3, b3 (fp32)

    def mlp(self, mode: int = binding.DSF_MODE_BF16_TC) -> binding.AttnMLP:
        return binding.AttnMLP(*self.mlp_t, mode=mode)

    @property
    def F(self) -> int:
        return self.tables.F


def table_to_device(t: np.ndarray, device) -> torch.Tensor:
    if t.dtype == np.uint16:
        return torch.from_numpy(t.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(t, dtype=np.float32)).to(device)


HASH_LOAD = 0.5  # keys per slot of the hash tables built here


def hash_table_for(batch, tabs, device):
    """The batch's hash-table features as one HashTable: key space f for
    feature f, every admitted key inserted with its row; None without any."""
    hk = getattr(batch, "hash_keys", None)
    if not hk:
        return None
    n = sum(int(k.size) for k in hk.values())
    key_space = [f if f in hk else -1 for f in range(len(tabs))]
    dtype = binding.DSF_BF16 if tabs[0].dtype == torch.bfloat16 else binding.DSF_F32
    ht = binding.HashTable(max(8, int(n / HASH_LOAD)), batch.D, dtype, key_space, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    for f, keys in hk.items():
        ht.insert(f, torch.from_numpy(np.ascontiguousarray(keys, np.int64)).to(device), tabs[f], status)
    if int(status.item()):
        raise RuntimeError("hash table build: status 0x%x" % int(status.item()))
    return ht


def to_device(batch, device="cuda") -> DeviceBatch:
    tabs = [table_to_device(t, device) for t in batch.tables]
    ht = hash_table_for(batch, tabs, device)
    mlp_t = [torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)
             for a in (batch.W1, batch.b1, batch.W2, batch.b2, batch.w3, batch.b3)]
    return DeviceBatch(
        B=batch.B, D=batch.D, max_len=batch.max_len, q_feat=tuple(batch.q_feat),
        seq_table=tuple(batch.seq_table),
        tables=binding.EmbeddingTables(tabs, getattr(batch, "pooling", None), ht),
        values=torch.from_numpy(np.ascontiguousarray(batch.values, np.int64)).to(device),
        lengths=torch.from_numpy(np.ascontiguousarray(batch.lengths, np.int32)).to(device),
        seq_values=torch.from_numpy(np.ascontiguousarray(batch.seq_values, np.int64)).to(device),
        seq_lengths=torch.from_numpy(np.ascontiguousarray(batch.seq_lengths, np.int32)).to(device),
        mlp_t=mlp_t)
