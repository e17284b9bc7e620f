"""Host-side checks of the seeded input generators."""
import numpy as np

from recsys_sparse_embedding_gb300 import synth


def test_ids_only_draw_matches_full_draw():
    full = synth.generate("taobao", seed=5, B=256)
    ids = synth.generate("taobao", seed=5, B=256, ids_only=True)
    assert ids.tables == []
    for name in ("values", "lengths", "seq_values", "seq_lengths"):
        assert np.array_equal(getattr(full, name), getattr(ids, name)), name
    rows = synth.WORKLOADS["taobao"].rows
    off = np.concatenate([[0], np.cumsum(ids.lengths)])
    for f in range(16):
        v = ids.values[off[f * 256]:off[(f + 1) * 256]]
        assert v.size == 0 or (v.min() >= 0 and v.max() < rows[f])
