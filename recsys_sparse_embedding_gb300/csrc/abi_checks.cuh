// Host-side argument checks shared by the C entry points (forward and
// backward): every pointer, size and mode a call takes is validated here
// before any CUDA call, and a failure is returned as a DSF_E* status.
#pragma once
#include <cstdint>

#include "dinsparse.h"
#include "fwd_kernel.cuh"
#include "hash.cuh"

namespace dsf {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline bool hashed(const dsf_tables* t, int f) { return t->hash && t->hash->key_space[f] >= 0; }

inline int check_tables(const dsf_tables* t) {
  if (!t || !t->table_ptrs || !t->table_rows) return DSF_EINVAL;
  if (t->F < 1 || t->F > DSF_MAX_TABLES) return DSF_EINVAL;
  if (t->D != 16 && t->D != 64) return DSF_EUNSUPPORTED;
  if (t->dtype != DSF_F32 && t->dtype != DSF_BF16) return DSF_EUNSUPPORTED;
  if (const dsf_hash* h = t->hash) {
    if (!h->key_space || h->D != t->D || h->dtype != t->dtype) return DSF_EINVAL;
    if (h->capacity < 1 || h->capacity > (1ll << 40)) return DSF_EINVAL;
    const hash::Layout L = hash::layout(h->capacity, h->D, t->dtype == DSF_BF16 ? 2 : 4);
    if (!h->workspace || !aligned(h->workspace, 256) || h->ws_bytes < L.total) return DSF_EWORKSPACE;
    for (int f = 0; f < t->F; ++f)
      if (h->key_space[f] < -1 || h->key_space[f] > hash::kMaxKeySpace) return DSF_EINVAL;
  }
  for (int f = 0; f < t->F; ++f) {
    if (t->pooling && t->pooling[f] != DSF_POOL_SUM && t->pooling[f] != DSF_POOL_MEAN) return DSF_EINVAL;
    if (hashed(t, f)) continue;
    if (!t->table_ptrs[f] || !aligned(t->table_ptrs[f], 16)) return DSF_EINVAL;
    if (t->table_rows[f] < 0) return DSF_EINVAL;
  }
  return DSF_OK;
}

inline int check_kjt(const dsf_kjt* k, int32_t B, int32_t F) {
  if (!k) return DSF_EINVAL;
  if (k->n_values < 0 || k->n_values > INT32_MAX) return DSF_EINVAL;
  if (B > 0 && F > 0 && (!k->lengths_dev || !aligned(k->lengths_dev, 4))) return DSF_EINVAL;
  if (k->n_values > 0 && (!k->values_dev || !aligned(k->values_dev, 8))) return DSF_EINVAL;
  return DSF_OK;
}

inline int check_seq(const dsf_seq* s, int32_t B) {
  if (!s) return DSF_EINVAL;
  if (s->n_per_key < 0 || s->n_per_key > INT32_MAX) return DSF_EINVAL;
  if (s->max_len < 1 || s->max_len > 65536) return DSF_EINVAL;
  if (B > 0 && (!s->lengths_dev || !aligned(s->lengths_dev, 4))) return DSF_EINVAL;
  if (s->n_per_key > 0 && (!s->values_dev || !aligned(s->values_dev, 8))) return DSF_EINVAL;
  return DSF_OK;
}

inline int check_mlp(const dsf_mlp* m, int32_t D) {
  if (!m || !m->W1 || !m->b1 || !m->W2 || !m->b2 || !m->w3 || !m->b3) return DSF_EINVAL;
  if (!aligned(m->b1, 16) || !aligned(m->b2, 16) || !aligned(m->w3, 16)) return DSF_EINVAL;
  if (m->K1 != 12 * D || m->N1 != kN1 || m->N2 != kN2) return DSF_EUNSUPPORTED;
  if (m->mode != DSF_MODE_BF16_TC && m->mode != DSF_MODE_FP32) return DSF_EINVAL;

  return DSF_OK;
}

}  // namespace dsf
