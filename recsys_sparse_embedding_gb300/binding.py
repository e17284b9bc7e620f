"""ctypes binding of libdinsparse.so (include/dinsparse.h).

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels. PyTorch supplies device memory and the stream. There is no CPU
fallback: if the library is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdinsparse.so")

DSF_F32, DSF_BF16 = 0, 1
DSF_MODE_BF16_TC, DSF_MODE_FP32 = 0, 1
DSF_OK, DSF_EINVAL, DSF_EUNSUPPORTED, DSF_ECUDA, DSF_EWORKSPACE = 0, 1, 2, 3, 4
FLAG_ID_RANGE = 0x01
FLAG_NEG_LENGTH = 0x02
FLAG_SEQ_TRUNC = 0x04
FLAG_COUNT = 0x08
FLAG_TIMEOUT = 0x10
FLAG_NOT_PREPARED = 0x20
FLAG_HASH = 0x40
FLAG_HASH_FULL = 0x80
FLAG_GRAD_LIST = 0x100

EXPORTS = ["dsf_workspace_bytes", "dsf_workspace_init", "dsf_prepare_mlp", "emb_bag_pool",
           "din_jagged_attn", "din_sparse_fwd", "dsf_status_string", "dsf_grid_size",
           "emb_bag_pool_noalloc", "dsf_towers_workspace_bytes", "dsf_prepare_towers", "ctr_towers_fwd",
           "dsf_hash_workspace_bytes", "dsf_hash_init", "dsf_hash_insert", "dsf_hash_find",
           "dsf_bwd_workspace_bytes", "din_sparse_bwd", "emb_adagrad_update", "dsf_read_status",
           "dsf_bwd_workspace_offsets"]

_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t


class CHash(ctypes.Structure):
    _fields_ = [("workspace", _vp), ("ws_bytes", _sz), ("capacity", _i64), ("D", _i32), ("dtype", _i32),
                ("key_space", _vp)]


class CMlpGrads(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("dW1", "db1", "dW2", "db2", "dw3", "db3")]


class CRowGrads(ctypes.Structure):
    _fields_ = [("grad", _vp), ("touched", _vp), ("list", _vp), ("count", _vp), ("list_cap", _i64)]


class CTables(ctypes.Structure):
    _fields_ = [("table_ptrs", _vp), ("table_rows", _vp), ("F", _i32), ("D", _i32), ("dtype", _i32),
                ("pooling", _vp), ("hash", _vp)]


class CKjt(ctypes.Structure):
    _fields_ = [("values_dev", _vp), ("n_values", _i64), ("lengths_dev", _vp)]


class CSeq(ctypes.Structure):
    _fields_ = [("values_dev", _vp), ("n_per_key", _i64), ("lengths_dev", _vp), ("max_len", _i32)]


class CMlp(ctypes.Structure):
    _fields_ = [("W1", _vp), ("b1", _vp), ("W2", _vp), ("b2", _vp), ("w3", _vp), ("b3", _vp),
                ("K1", _i32), ("N1", _i32), ("N2", _i32), ("mode", _i32)]


class DsfError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (where, status_string(code), code))


_lib = None


def lib() -> ctypes.CDLL:
    """Loads libdinsparse.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libdinsparse.so is not built (run recsys_sparse_embedding_gb300"
                               ".build.build()); there is no fallback implementation")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER
        L.dsf_workspace_bytes.argtypes = [_i32, _i32]
        L.dsf_workspace_bytes.restype = _sz
        L.dsf_workspace_init.argtypes = [_vp, _sz, _vp]
        L.dsf_workspace_init.restype = ctypes.c_int
        L.dsf_prepare_mlp.argtypes = [P(CMlp), _i32, _vp, _sz, _vp]
        L.dsf_prepare_mlp.restype = ctypes.c_int
        L.emb_bag_pool.argtypes = [P(CTables), P(CKjt), _i32, _vp, _vp, _sz, _vp, _vp]
        L.emb_bag_pool.restype = ctypes.c_int
        L.din_jagged_attn.argtypes = [P(CTables), P(CKjt), P(CSeq), _vp, _vp, _i32, P(CMlp),
                                      _vp, _vp, _vp, _sz, _vp, _vp]
        L.din_jagged_attn.restype = ctypes.c_int
        L.din_sparse_fwd.argtypes = [P(CTables), P(CKjt), P(CSeq), _vp, _vp, _i32, P(CMlp),
                                     _vp, _vp, _vp, _vp, _sz, _vp, _vp]
        L.din_sparse_fwd.restype = ctypes.c_int
        L.dsf_status_string.argtypes = [ctypes.c_int]
        L.dsf_status_string.restype = ctypes.c_char_p
        L.emb_bag_pool_noalloc.argtypes = [P(CTables), P(CKjt), _i32, _vp, _vp, _vp]
        L.emb_bag_pool_noalloc.restype = ctypes.c_int
        L.dsf_grid_size.argtypes = [_i32, _i32, _i32, _i32]
        L.dsf_grid_size.restype = _i32
        L.dsf_towers_workspace_bytes.argtypes = []
        L.dsf_towers_workspace_bytes.restype = _sz
        L.dsf_prepare_towers.argtypes = [P(CTowers), _vp, _sz, _vp]
        L.dsf_prepare_towers.restype = ctypes.c_int
        L.ctr_towers_fwd.argtypes = [_vp, _vp, _i32, P(CTowers), _vp, _vp, _sz, _vp, _vp]
        L.ctr_towers_fwd.restype = ctypes.c_int
        L.dsf_hash_workspace_bytes.argtypes = [_i64, _i32, _i32]
        L.dsf_hash_workspace_bytes.restype = _sz
        L.dsf_hash_init.argtypes = [P(CHash), _vp]
        L.dsf_hash_init.restype = ctypes.c_int
        L.dsf_hash_insert.argtypes = [P(CHash), _i32, _vp, _vp, _i64, _vp, _vp]
        L.dsf_hash_insert.restype = ctypes.c_int
        L.dsf_hash_find.argtypes = [P(CHash), _i32, _vp, _i64, _vp, _vp, _vp]
        L.dsf_hash_find.restype = ctypes.c_int
        L.dsf_bwd_workspace_bytes.argtypes = [_i32, _i64, _i64, _i32]
        L.dsf_bwd_workspace_bytes.restype = _sz
        L.din_sparse_bwd.argtypes = [P(CTables), P(CKjt), P(CSeq), _vp, _vp, _i32, P(CMlp), _vp, _vp, _vp,
                                     P(CMlpGrads), P(CRowGrads), _vp, _sz, _vp, _vp]
        L.din_sparse_bwd.restype = ctypes.c_int
        L.emb_adagrad_update.argtypes = [P(CTables), _vp, P(CRowGrads), ctypes.c_float, ctypes.c_float, _vp, _vp]
        L.emb_adagrad_update.restype = ctypes.c_int
        L.dsf_read_status.argtypes = [_vp, _vp, _vp]
        L.dsf_read_status.restype = ctypes.c_int
        L.dsf_bwd_workspace_offsets.argtypes = [_i32, _i64, _i64, _i32, _vp]
        L.dsf_bwd_workspace_offsets.restype = ctypes.c_int
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().dsf_status_string(int(code)).decode()


def read_status(status, stream=None) -> int:
    """The DSF_FLAG_* bits in a device status word, once the work queued on
    the stream so far has finished (dsf_read_status)."""
    out = ctypes.c_int32(0)
    _check(lib().dsf_read_status(_dptr(status), ctypes.byref(out), _stream_ptr(stream)), "dsf_read_status")
    return int(out.value)


def _check(rc: int, where: str) -> None:
    if rc != DSF_OK:
        raise DsfError(rc, where)


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


class EmbeddingTables:
    """F device tables [rows_f, D], all fp32 or all bf16. pooling: per table
    DSF_POOL_SUM or DSF_POOL_MEAN (None: all sum)."""

    def __init__(self, tables: Sequence[torch.Tensor], pooling: Optional[Sequence[int]] = None,
                 hash_table: Optional["HashTable"] = None):
        self.tables = list(tables)
        self.hash = hash_table
        F = len(self.tables)
        D = int(self.tables[0].shape[1])
        dt = self.tables[0].dtype
        for t in self.tables:
            if t.dim() != 2 or int(t.shape[1]) != D or t.dtype != dt or not t.is_contiguous():
                raise ValueError("tables must be contiguous [rows, D] with one D and dtype")
        self.F, self.D = F, D
        self.dtype = DSF_BF16 if dt == torch.bfloat16 else DSF_F32
        self._ptrs = (ctypes.c_void_p * F)(*[t.data_ptr() for t in self.tables])
        self._rows = (ctypes.c_int64 * F)(*[int(t.shape[0]) for t in self.tables])
        self.pooling = None if pooling is None else [int(x) for x in pooling]
        if self.pooling is not None and len(self.pooling) != F:
            raise ValueError("pooling needs one mode per table")
        self._pool = None if self.pooling is None else (ctypes.c_int32 * F)(*self.pooling)
        self.c = CTables(ctypes.cast(self._ptrs, _vp), ctypes.cast(self._rows, _vp), F, D, self.dtype,
                         None if self._pool is None else ctypes.cast(self._pool, _vp),
                         None if hash_table is None else ctypes.cast(ctypes.pointer(hash_table.c), _vp))
        if hash_table is not None and len(hash_table.key_space) != F:
            raise ValueError("the hash table needs one key space entry per table")

    @property
    def rows(self):
        return [int(t.shape[0]) for t in self.tables]


class AttnMLP:
    """Device fp32 attention MLP in Linear [out, in] layout."""

    def __init__(self, W1, b1, W2, b2, w3, b3, mode: int = DSF_MODE_BF16_TC):
        self.t = [x.contiguous() for x in (W1, b1, W2, b2, w3.reshape(-1), b3.reshape(-1))]
        W1, b1, W2, b2, w3, b3 = self.t
        self.mode = int(mode)
        self.c = CMlp(W1.data_ptr(), b1.data_ptr(), W2.data_ptr(), b2.data_ptr(), w3.data_ptr(),
                      b3.data_ptr(), int(W1.shape[1]), int(W1.shape[0]), int(W2.shape[0]), self.mode)

    def with_mode(self, mode: int) -> "AttnMLP":
        return AttnMLP(*self.t, mode=mode)


class Workspace:
    """Caller-owned scratch for one stream: grid-barrier state, per-CTA partial
    sums, packed MLP weights and the query buffer."""

    def __init__(self, B: int, D: int, device=None, stream=None):
        n = int(lib().dsf_workspace_bytes(int(B), int(D)))
        if n == 0:
            raise DsfError(DSF_EUNSUPPORTED, "dsf_workspace_bytes")
        self.B, self.D, self.nbytes = int(B), int(D), n
        self.buf = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
        _check(lib().dsf_workspace_init(self.buf.data_ptr(), n, _stream_ptr(stream)),
               "dsf_workspace_init")

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    def prepare(self, mlp: AttnMLP, stream=None) -> None:
        _check(lib().dsf_prepare_mlp(ctypes.byref(mlp.c), self.D, self.ptr, self.nbytes,
                                     _stream_ptr(stream)), "dsf_prepare_mlp")


def _kjt(values: torch.Tensor, lengths: torch.Tensor) -> CKjt:
    return CKjt(values.data_ptr(), int(values.numel()), lengths.data_ptr())


def _seq(seq_values: torch.Tensor, seq_lengths: torch.Tensor, max_len: int) -> CSeq:
    n = int(seq_values.shape[-1]) if seq_values.dim() == 2 else int(seq_values.numel()) // 3
    return CSeq(seq_values.data_ptr(), n, seq_lengths.data_ptr(), int(max_len))


def _i3(x) -> ctypes.Array:
    return (ctypes.c_int32 * 3)(*[int(v) for v in x])


def emb_bag_pool(tables: EmbeddingTables, values: torch.Tensor, lengths: torch.Tensor, B: int,
                 pooled: torch.Tensor, workspace: Workspace, status: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    kjt = _kjt(values, lengths)
    _check(lib().emb_bag_pool(ctypes.byref(tables.c), ctypes.byref(kjt), int(B), pooled.data_ptr(),
                              workspace.ptr, workspace.nbytes, _dptr(status), _stream_ptr(stream)),
           "emb_bag_pool")
    return pooled


def emb_bag_pool_noalloc(tables: EmbeddingTables, values: torch.Tensor, lengths: torch.Tensor,
                         B: int, pooled: torch.Tensor, status: Optional[torch.Tensor] = None,
                         stream=None) -> torch.Tensor:
    """emb_bag_pool without a workspace, for callers that cannot allocate
    device memory; its scratch is a fixed array inside the library."""
    kjt = _kjt(values, lengths)
    _check(lib().emb_bag_pool_noalloc(ctypes.byref(tables.c), ctypes.byref(kjt), int(B),
                                      pooled.data_ptr(), _dptr(status), _stream_ptr(stream)),
           "emb_bag_pool_noalloc")
    return pooled


def din_jagged_attn(tables: EmbeddingTables, values: torch.Tensor, lengths: torch.Tensor,
                    seq_values: torch.Tensor, seq_lengths: torch.Tensor, max_len: int,
                    q_feat, seq_table, B: int, mlp: AttnMLP, din: torch.Tensor,
                    workspace: Workspace, logits: Optional[torch.Tensor] = None,
                    status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    kjt, seq = _kjt(values, lengths), _seq(seq_values, seq_lengths, max_len)
    qf, st = _i3(q_feat), _i3(seq_table)
    _check(lib().din_jagged_attn(ctypes.byref(tables.c), ctypes.byref(kjt), ctypes.byref(seq),
                                 ctypes.cast(qf, _vp), ctypes.cast(st, _vp), int(B),
                                 ctypes.byref(mlp.c), din.data_ptr(), _dptr(logits), workspace.ptr,
                                 workspace.nbytes, _dptr(status), _stream_ptr(stream)),
           "din_jagged_attn")
    return din


def din_sparse_fwd(tables: EmbeddingTables, values: torch.Tensor, lengths: torch.Tensor,
                   seq_values: torch.Tensor, seq_lengths: torch.Tensor, max_len: int,
                   q_feat, seq_table, B: int, mlp: AttnMLP, pooled: torch.Tensor,
                   din: torch.Tensor, workspace: Workspace, logits: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None, stream=None):
    kjt, seq = _kjt(values, lengths), _seq(seq_values, seq_lengths, max_len)
    qf, st = _i3(q_feat), _i3(seq_table)
    _check(lib().din_sparse_fwd(ctypes.byref(tables.c), ctypes.byref(kjt), ctypes.byref(seq),
                                ctypes.cast(qf, _vp), ctypes.cast(st, _vp), int(B),
                                ctypes.byref(mlp.c), pooled.data_ptr(), din.data_ptr(),
                                _dptr(logits), workspace.ptr, workspace.nbytes, _dptr(status),
                                _stream_ptr(stream)),
           "din_sparse_fwd")
    return pooled, din


def grid_size(D: int, dtype: int, mode: int, with_attention: bool) -> int:
    return int(lib().dsf_grid_size(int(D), int(dtype), int(mode), int(bool(with_attention))))


class CTowers(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("Wd1", "bd1", "Wd2", "bd2", "Wd3", "bd3", "Wf1", "bf1", "wo", "bo")]


class Towers:
    """The dense towers' device fp32 weights ([out, in]) and their packed
    workspace. Wd1 [512, 256], bd1 [512], Wd2 [256, 512], bd2 [256],
    Wd3 [128, 256], bd3 [128], Wf1 [64, 176], bf1 [64], wo [64], bo [1]."""

    NAMES = ("Wd1", "bd1", "Wd2", "bd2", "Wd3", "bd3", "Wf1", "bf1", "wo", "bo")

    def __init__(self, weights: Sequence[torch.Tensor], device="cuda"):
        self.w = [torch.as_tensor(t, dtype=torch.float32, device=device).contiguous() for t in weights]
        if len(self.w) != len(self.NAMES):
            raise ValueError("towers need %d weight tensors" % len(self.NAMES))
        self.c = CTowers(*[t.data_ptr() for t in self.w])
        self.nbytes = int(lib().dsf_towers_workspace_bytes())
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)

    def prepare(self, stream=None):
        _check(lib().dsf_prepare_towers(ctypes.byref(self.c), self.buf.data_ptr(), self.nbytes,
                                        _stream_ptr(stream)), "dsf_prepare_towers")


def ctr_towers_fwd(pooled: torch.Tensor, din: torch.Tensor, B: int, towers: Towers,
                   logit: torch.Tensor, status: Optional[torch.Tensor] = None, stream=None):
    _check(lib().ctr_towers_fwd(pooled.data_ptr(), din.data_ptr(), int(B), ctypes.byref(towers.c),
                                logit.data_ptr(), towers.buf.data_ptr(), towers.nbytes,
                                _dptr(status), _stream_ptr(stream)), "ctr_towers_fwd")
    return logit


class HashTable:
    """Hash-table storage (one device workspace) for the tables whose
    key_space[f] >= 0: raw int64 keys in [0, 2^56) map to rows of one fused
    pool; an unseen key reads zero. capacity: the minimum slot count."""

    def __init__(self, capacity: int, D: int, dtype: int, key_space: Sequence[int], device="cuda",
                 stream=None):
        self.key_space = [int(k) for k in key_space]
        self._ks = (ctypes.c_int32 * len(self.key_space))(*self.key_space)
        self.nbytes = int(lib().dsf_hash_workspace_bytes(int(capacity), int(D), int(dtype)))
        if self.nbytes == 0:
            raise DsfError(DSF_EINVAL, "dsf_hash_workspace_bytes")
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.c = CHash(self.buf.data_ptr(), self.nbytes, int(capacity), int(D), int(dtype),
                       ctypes.cast(self._ks, _vp))
        _check(lib().dsf_hash_init(ctypes.byref(self.c), _stream_ptr(stream)), "dsf_hash_init")

    def insert(self, key_space: int, keys: torch.Tensor, rows: torch.Tensor,
               status: Optional[torch.Tensor] = None, stream=None):
        keys = keys.contiguous()
        rows = rows.contiguous()
        _check(lib().dsf_hash_insert(ctypes.byref(self.c), int(key_space), keys.data_ptr(), rows.data_ptr(),
                                     int(keys.numel()), _dptr(status), _stream_ptr(stream)),
               "dsf_hash_insert")

    def find(self, key_space: int, keys: torch.Tensor, status: Optional[torch.Tensor] = None,
             stream=None) -> torch.Tensor:
        keys = keys.contiguous()
        out = torch.empty_like(keys)
        _check(lib().dsf_hash_find(ctypes.byref(self.c), int(key_space), keys.data_ptr(), int(keys.numel()),
                                   out.data_ptr(), _dptr(status), _stream_ptr(stream)), "dsf_hash_find")
        return out


class MlpGrads:
    """Device fp32 gradients of the attention MLP (overwritten by a backward
    call): dW1 [256, 12D], db1 [256], dW2 [64, 256], db2 [64], dw3 [64], db3 [1]."""

    def __init__(self, D: int, device="cuda"):
        K1 = 12 * D
        self.t = dict(dW1=torch.zeros(256, K1, device=device), db1=torch.zeros(256, device=device),
                      dW2=torch.zeros(64, 256, device=device), db2=torch.zeros(64, device=device),
                      dw3=torch.zeros(64, device=device), db3=torch.zeros(1, device=device))
        self.c = CMlpGrads(*[self.t[n].data_ptr() for n in ("dW1", "db1", "dW2", "db2", "dw3", "db3")])

    def __getitem__(self, k):
        return self.t[k]


class SparseState:
    """Per-storage row-gradient buffers, touched flags and AdaGrad
    accumulators for a set of tables: one [rows, D] / [rows] set per plain
    table, and one for the hash pool shared by the hash-table tables; the
    touched-row list holds list_cap entries."""

    def __init__(self, tables: EmbeddingTables, list_cap: int, device="cuda", accum_init: float = 0.0):
        F, D = tables.F, tables.D
        ks = tables.hash.key_space if tables.hash is not None else [-1] * F
        pool_rows = None
        if tables.hash is not None:
            pool_rows = (self._pool_rows(tables.hash))
        first = next((f for f in range(F) if ks[f] >= 0), None)
        self.grad, self.touched, self.accum = [], [], []
        for f in range(F):
            if ks[f] >= 0 and f != first:
                self.grad.append(self.grad[first])
                self.touched.append(self.touched[first])
                self.accum.append(self.accum[first])
                continue
            n = pool_rows if ks[f] >= 0 else int(tables.tables[f].shape[0])
            self.grad.append(torch.zeros(n, D, device=device))
            self.touched.append(torch.zeros(n, dtype=torch.int32, device=device))
            self.accum.append(torch.full((n, D), float(accum_init), device=device))
        self.list = torch.zeros(max(1, int(list_cap)), dtype=torch.int64, device=device)
        self.count = torch.zeros(1, dtype=torch.int32, device=device)
        self._g = (_vp * F)(*[t.data_ptr() for t in self.grad])
        self._t = (_vp * F)(*[t.data_ptr() for t in self.touched])
        self._a = (_vp * F)(*[t.data_ptr() for t in self.accum])
        self.c = CRowGrads(ctypes.cast(self._g, _vp), ctypes.cast(self._t, _vp), self.list.data_ptr(),
                           self.count.data_ptr(), int(list_cap))

    @staticmethod
    def _pool_rows(ht: "HashTable") -> int:
        slots = 8
        while slots < ht.c.capacity:
            slots *= 2
        return slots + 1

    @property
    def accum_ptrs(self):
        return ctypes.cast(self._a, _vp)


class BwdWorkspace:
    def __init__(self, B: int, n_values: int, n_per_key: int, D: int, device="cuda"):
        self.nbytes = int(lib().dsf_bwd_workspace_bytes(int(B), int(n_values), int(n_per_key), int(D)))
        if self.nbytes == 0:
            raise DsfError(DSF_EINVAL, "dsf_bwd_workspace_bytes")
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        off = (ctypes.c_int64 * 6)()
        _check(lib().dsf_bwd_workspace_offsets(int(B), int(n_values), int(n_per_key), int(D),
                                               ctypes.cast(off, _vp)), "dsf_bwd_workspace_offsets")
        self.offsets = list(off)
        self.D = int(D)

    def views(self, P: int, bf16: bool):
        """The intermediates the last din_sparse_bwd left in this workspace,
        over the first P positions: x, h1, h2 (h1 W2^T), dh2, g (dh2 W2),
        dh1, as tensors viewing the buffer."""
        K1 = 12 * self.D
        op = torch.bfloat16 if bf16 else torch.float32
        out = {}
        for i, (name, width, dt) in enumerate((("x", K1, op), ("h1", 256, op), ("h2", 64, torch.float32),
                                               ("dh2", 64, op), ("g", 256, torch.float32), ("dh1", 256, op))):
            es = 2 if dt == torch.bfloat16 else 4
            o = self.offsets[i]
            out[name] = self.buf[o:o + P * width * es].view(dt).view(P, width)
        return out


def din_sparse_bwd(tables: EmbeddingTables, values, lengths, seq_values, seq_lengths, max_len: int, q_feat,
                   seq_table, B: int, mlp: AttnMLP, pooled, dpooled, ddin, grads: MlpGrads,
                   state: SparseState, ws: BwdWorkspace, status=None, stream=None):
    kjt = _kjt(values, lengths)
    seq = _seq(seq_values, seq_lengths, max_len)
    qf = (ctypes.c_int32 * 3)(*q_feat)
    st = (ctypes.c_int32 * 3)(*seq_table)
    _check(lib().din_sparse_bwd(ctypes.byref(tables.c), ctypes.byref(kjt), ctypes.byref(seq),
                                ctypes.cast(qf, _vp), ctypes.cast(st, _vp), int(B), ctypes.byref(mlp.c),
                                pooled.data_ptr(), _dptr(dpooled), ddin.data_ptr(), ctypes.byref(grads.c),
                                ctypes.byref(state.c), ws.buf.data_ptr(), ws.nbytes, _dptr(status),
                                _stream_ptr(stream)), "din_sparse_bwd")


def emb_adagrad_update(tables: EmbeddingTables, state: SparseState, lr: float = 1e-3, eps: float = 1e-10,
                       status=None, stream=None):
    _check(lib().emb_adagrad_update(ctypes.byref(tables.c), state.accum_ptrs, ctypes.byref(state.c),
                                    float(lr), float(eps), _dptr(status), _stream_ptr(stream)),
           "emb_adagrad_update")
