"""Host-side checks of the C ABI: the library builds and loads, exports every
function include/dinsparse.h declares, and rejects bad arguments before any
CUDA call (these run without a GPU)."""
import ctypes
import os
import re

import pytest

from recsys_sparse_embedding_gb300 import binding
from recsys_sparse_embedding_gb300 import build as nbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    nbuild.build()
    return binding.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dinsparse.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_function(L):
    names = declared_functions()
    assert set(binding.EXPORTS) <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_workspace_bytes(L):
    assert L.dsf_workspace_bytes(8192, 16) > 8192 * 48 * 4
    assert L.dsf_workspace_bytes(8192, 32) == 0
    assert L.dsf_workspace_bytes(0, 64) > 0


def _tables(F=16, D=16, dtype=0, ptr=4096):
    ptrs = (ctypes.c_void_p * F)(*([ptr] * F))
    rows = (ctypes.c_int64 * F)(*([10] * F))
    return binding.CTables(ctypes.cast(ptrs, ctypes.c_void_p), ctypes.cast(rows, ctypes.c_void_p),
                           F, D, dtype), (ptrs, rows)


def test_emb_bag_pool_rejects_bad_arguments(L):
    t, keep = _tables()
    k = binding.CKjt(4096, 16, 4096)
    P = ctypes.byref
    assert L.emb_bag_pool(None, P(k), 1, 4096, 4096, 1 << 30, None, None) == binding.DSF_EINVAL
    assert L.emb_bag_pool(P(t), P(k), -1, 4096, 4096, 1 << 30, None, None) == binding.DSF_EINVAL
    assert L.emb_bag_pool(P(t), P(k), 1, None, 4096, 1 << 30, None, None) == binding.DSF_EINVAL
    assert L.emb_bag_pool(P(t), P(k), 1, 4096, None, 1 << 30, None, None) == binding.DSF_EWORKSPACE
    assert L.emb_bag_pool(P(t), P(k), 1, 4096, 4096 + 16, 1 << 30, None, None) == binding.DSF_EWORKSPACE
    assert L.emb_bag_pool(P(t), P(k), 1, 4096, 4096, 64, None, None) == binding.DSF_EWORKSPACE
    bad, keep2 = _tables(D=32)
    assert L.emb_bag_pool(P(bad), P(k), 1, 4096, 4096, 1 << 30, None, None) == binding.DSF_EUNSUPPORTED
    bad, keep3 = _tables(F=33)
    assert L.emb_bag_pool(P(bad), P(k), 1, 4096, 4096, 1 << 30, None, None) == binding.DSF_EINVAL
    bad, keep4 = _tables(ptr=4100)   # misaligned table
    assert L.emb_bag_pool(P(bad), P(k), 1, 4096, 4096, 1 << 30, None, None) == binding.DSF_EINVAL
    neg = binding.CKjt(4096, -1, 4096)
    assert L.emb_bag_pool(P(t), P(neg), 1, 4096, 4096, 1 << 30, None, None) == binding.DSF_EINVAL
    # B = 0 is a valid no-op and touches no device
    assert L.emb_bag_pool(P(t), P(k), 0, 4096, 4096, 1 << 30, None, None) == binding.DSF_OK


def test_attention_rejects_bad_arguments(L):
    t, keep = _tables()
    k = binding.CKjt(4096, 16, 4096)
    s = binding.CSeq(4096, 10, 4096, 100)
    m = binding.CMlp(4096, 4096, 4096, 4096, 4096, 4096, 192, 256, 64, 0)
    q = (ctypes.c_int32 * 3)(1, 5, 2)
    P = ctypes.byref
    args = lambda **kw: dict(dict(t=P(t), k=P(k), s=P(s), q=q, st=q, B=4, m=P(m), din=4096), **kw)

    def call(**kw):
        a = args(**kw)
        return L.din_jagged_attn(a["t"], a["k"], a["s"], ctypes.cast(a["q"], ctypes.c_void_p),
                                 ctypes.cast(a["st"], ctypes.c_void_p), a["B"], a["m"], a["din"],
                                 None, 4096, 1 << 30, None, None)
    assert call(q=(ctypes.c_int32 * 3)(1, 5, 16)) == binding.DSF_EINVAL
    assert call(st=(ctypes.c_int32 * 3)(-1, 5, 2)) == binding.DSF_EINVAL
    assert call(din=None) == binding.DSF_EINVAL
    assert call(din=4100) == binding.DSF_EINVAL
    bad_seq = binding.CSeq(4096, 10, 4096, 0)
    assert call(s=P(bad_seq)) == binding.DSF_EINVAL
    bad_mlp = binding.CMlp(4096, 4096, 4096, 4096, 4096, 4096, 191, 256, 64, 0)
    assert call(m=P(bad_mlp)) == binding.DSF_EUNSUPPORTED
    null_mlp = binding.CMlp(None, 4096, 4096, 4096, 4096, 4096, 192, 256, 64, 0)
    assert call(m=P(null_mlp)) == binding.DSF_EINVAL
    assert call(B=0) == binding.DSF_OK
    assert L.din_sparse_fwd(P(t), P(k), P(s), ctypes.cast(q, ctypes.c_void_p),
                            ctypes.cast(q, ctypes.c_void_p), 4, P(m), None, 4096, None, 4096,
                            1 << 30, None, None) == binding.DSF_EINVAL


def test_towers_reject_bad_arguments(L):
    w = binding.CTowers(*([4096] * 10))
    P = ctypes.byref
    n = L.dsf_towers_workspace_bytes()
    assert n >= (512 * 256 + 256 * 512 + 128 * 256 + 64 * 192) * 2

    def call(pooled=4096, din=4096, B=4, tw=P(w), logit=4096, ws=4096, nb=n):
        return L.ctr_towers_fwd(pooled, din, B, tw, logit, ws, nb, None, None)
    assert call(B=-1) == binding.DSF_EINVAL
    assert call(tw=None) == binding.DSF_EINVAL
    assert call(pooled=None) == binding.DSF_EINVAL
    assert call(din=4100) == binding.DSF_EINVAL
    assert call(logit=None) == binding.DSF_EINVAL
    assert call(tw=P(binding.CTowers(*([4096] * 9 + [0])))) == binding.DSF_EINVAL
    assert call(ws=None) == binding.DSF_EWORKSPACE
    assert call(ws=4096 + 16) == binding.DSF_EWORKSPACE
    assert call(nb=n - 1) == binding.DSF_EWORKSPACE
    assert call(B=0) == binding.DSF_OK
    assert L.dsf_prepare_towers(None, 4096, n, None) == binding.DSF_EINVAL
    assert L.dsf_prepare_towers(P(w), 4096, n - 1, None) == binding.DSF_EWORKSPACE


def test_hash_entry_points_reject_bad_arguments(L):
    P = ctypes.byref
    n = L.dsf_hash_workspace_bytes(1000, 16, 0)
    # 1000 slots round up to 1024 = 128 buckets of 8: keys, then 1025 rows
    assert n == 256 + 1024 * 8 + ((1025 * 64 + 255) // 256) * 256
    assert L.dsf_hash_workspace_bytes(0, 16, 0) == 0
    assert L.dsf_hash_workspace_bytes(8, 32, 0) == 0
    assert L.dsf_hash_workspace_bytes(8, 16, 2) == 0
    ks = (ctypes.c_int32 * 16)(*([-1] * 16))
    ok = binding.CHash(4096, n, 1000, 16, 0, ctypes.cast(ks, ctypes.c_void_p))
    assert L.dsf_hash_init(None, None) == binding.DSF_EINVAL
    assert L.dsf_hash_init(P(binding.CHash(4096, n - 1, 1000, 16, 0, None)), None) == binding.DSF_EWORKSPACE
    assert L.dsf_hash_init(P(binding.CHash(4100, n, 1000, 16, 0, None)), None) == binding.DSF_EWORKSPACE
    assert L.dsf_hash_init(P(binding.CHash(4096, n, 1000, 24, 0, None)), None) == binding.DSF_EUNSUPPORTED
    assert L.dsf_hash_insert(P(ok), 255, 4096, 4096, 4, None, None) == binding.DSF_EINVAL
    assert L.dsf_hash_insert(P(ok), -1, 4096, 4096, 4, None, None) == binding.DSF_EINVAL
    assert L.dsf_hash_insert(P(ok), 0, 4096, 4100, 4, None, None) == binding.DSF_EINVAL
    assert L.dsf_hash_insert(P(ok), 0, 4096, 4096, 0, None, None) == binding.DSF_OK
    assert L.dsf_hash_find(P(ok), 0, 4096, 4, None, None, None) == binding.DSF_EINVAL
    assert L.dsf_hash_find(P(ok), 0, 4096, 0, None, None, None) == binding.DSF_OK
    # the tables' view of the hash storage: key spaces, D and the workspace
    t, keep = _tables()
    k = binding.CKjt(4096, 16, 4096)

    def pool_with(h):
        t.hash = ctypes.cast(ctypes.pointer(h), ctypes.c_void_p)
        return L.emb_bag_pool(P(t), P(k), 1, 4096, 4096, 1 << 30, None, None)
    bad_ks = (ctypes.c_int32 * 16)(*([255] + [-1] * 15))
    assert pool_with(binding.CHash(4096, n, 1000, 16, 0, ctypes.cast(bad_ks, ctypes.c_void_p))) == binding.DSF_EINVAL
    assert pool_with(binding.CHash(4096, n, 1000, 64, 0, ctypes.cast(ks, ctypes.c_void_p))) == binding.DSF_EINVAL
    assert pool_with(binding.CHash(4096, n, 1000, 16, 0, None)) == binding.DSF_EINVAL
    assert pool_with(binding.CHash(4096, n - 256, 1000, 16, 0, ctypes.cast(ks, ctypes.c_void_p))) == \
        binding.DSF_EWORKSPACE
    # a hashed table's own pointer is ignored (null is fine)
    ptrs = (ctypes.c_void_p * 16)(*([None] + [4096] * 15))
    t.table_ptrs = ctypes.cast(ptrs, ctypes.c_void_p)
    one = (ctypes.c_int32 * 16)(*([0] + [-1] * 15))
    t.hash = ctypes.cast(ctypes.pointer(binding.CHash(4096, n, 1000, 16, 0, ctypes.cast(one, ctypes.c_void_p))),
                         ctypes.c_void_p)
    assert L.emb_bag_pool(P(t), P(k), 0, 4096, 4096, 1 << 30, None, None) == binding.DSF_OK
    t.hash = None
    assert L.emb_bag_pool(P(t), P(k), 1, 4096, 4096, 1 << 30, None, None) == binding.DSF_EINVAL


def test_status_strings(L):
    for code in range(5):
        assert binding.status_string(code)
    assert binding.status_string(99) == "unknown status"


def test_no_fallback_when_library_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        binding.lib()


def test_read_status_rejects_null_pointers(L):
    out = ctypes.c_int32(7)
    assert L.dsf_read_status(None, ctypes.byref(out), None) == binding.DSF_EINVAL
    assert L.dsf_read_status(4096, None, None) == binding.DSF_EINVAL
    assert out.value == 7


def test_bwd_workspace_offsets(L):
    """The six intermediates lie inside the workspace, 256-byte aligned, each
    with room for its [n_per_key, width] fp32 rows, without overlap."""
    for B, nv, npk, D in ((8192, 200000, 40000, 16), (3, 0, 0, 64), (0, 5, 7, 16)):
        off = (ctypes.c_int64 * 6)()
        assert L.dsf_bwd_workspace_offsets(B, nv, npk, D, off) == binding.DSF_OK
        total = L.dsf_bwd_workspace_bytes(B, nv, npk, D)
        widths = (12 * D, 256, 64, 64, 256, 256)
        spans = sorted((off[i], off[i] + npk * widths[i] * 4) for i in range(6))
        for (a, e), (a2, _) in zip(spans, spans[1:]):
            assert e <= a2
        assert all(o % 256 == 0 for o in off) and spans[-1][1] <= total
    off = (ctypes.c_int64 * 6)()
    assert L.dsf_bwd_workspace_offsets(4, 1, 1, 32, off) == binding.DSF_EINVAL
    assert L.dsf_bwd_workspace_offsets(4, -1, 1, 16, off) == binding.DSF_EINVAL
    assert L.dsf_bwd_workspace_offsets(4, 1, 1, 16, None) == binding.DSF_EINVAL
