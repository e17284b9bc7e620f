"""GB300-native (sm_103a) MultiTowerDIN sparse forward.

The compute lives in libdinsparse.so (CUDA kernels behind the C ABI in
include/dinsparse.h); this package is its Python binding, the build script and
the seeded workload generator.
"""
from .binding import (AttnMLP, DsfError, EmbeddingTables, Workspace, din_jagged_attn,  # noqa: F401
                      din_sparse_fwd, emb_bag_pool, grid_size, lib, status_string)
