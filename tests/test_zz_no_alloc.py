"""emb_bag_pool_noalloc: pooling for callers that cannot allocate device memory
(for example a serving runtime whose device memory belongs to its own arena, or
code running under stream capture, where cudaMalloc is not allowed). Its only
scratch is a fixed array inside the library, so it must give exactly what the
workspace-based emb_bag_pool gives, call after call. This file is collected
last on purpose; it passes alone in a fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

import oracle
from recsys_sparse_embedding_gb300 import binding, synth
from recsys_sparse_embedding_gb300.device_batch import to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl,B", [("taobao", 3000), ("long_multihot", 700), ("wide_bf16", 300)])
def test_noalloc_matches_workspace_pooling_twice(wl, B):
    batch = synth.generate(wl, seed=7, B=B)
    db = to_device(batch)
    ws = binding.Workspace(batch.B, batch.D)
    ref = torch.full((batch.B, db.F * db.D), float("nan"), device="cuda")
    st_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.emb_bag_pool(db.tables, db.values, db.lengths, batch.B, ref, ws, status=st_ref)
    torch.cuda.synchronize()
    want = ref.cpu().numpy()
    assert int(st_ref.item()) == 0
    # the pooling the oracle gives, summed in the same bag order: bit-exact
    assert np.array_equal(want, oracle.pool_batch(batch)[0])
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        binding.emb_bag_pool_noalloc(db.tables, db.values, db.lengths, batch.B, out, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        # same kernel, same bag order: the sums are identical, not merely close
        assert np.array_equal(out.cpu().numpy(), want)


def test_noalloc_rejects_bad_arguments_without_launching():
    batch = synth.generate("tiny", seed=1)
    db = to_device(batch)
    out = torch.empty(batch.B, db.F * db.D, device="cuda")
    with pytest.raises(binding.DsfError):
        binding.emb_bag_pool_noalloc(db.tables, db.values, db.lengths, -1, out)


def test_noalloc_captured_in_a_graph():
    """One eager call (it looks up and clears the array), then two calls
    captured into one CUDA graph, replayed twice: both outputs equal the
    workspace-based pooling and the oracle's, status zero."""
    batch = synth.generate("taobao", seed=8, B=2000)
    db = to_device(batch)
    ws = binding.Workspace(batch.B, batch.D)
    ref = torch.empty(batch.B, db.F * db.D, device="cuda")
    binding.emb_bag_pool(db.tables, db.values, db.lengths, batch.B, ref, ws)
    torch.cuda.synchronize()
    want = ref.cpu().numpy()
    assert np.array_equal(want, oracle.pool_batch(batch)[0])
    outs = [torch.full_like(ref, float("nan")) for _ in range(2)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.emb_bag_pool_noalloc(db.tables, db.values, db.lengths, batch.B, outs[0], status=st)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for o in outs:
            binding.emb_bag_pool_noalloc(db.tables, db.values, db.lengths, batch.B, o, status=st)
    for _ in range(2):
        for o in outs:
            o.fill_(float("nan"))
        st.zero_()
        g.replay()
        assert binding.read_status(st) == 0
        for o in outs:
            assert np.array_equal(o.cpu().numpy(), want)
