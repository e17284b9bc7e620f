// Hash-table workspace: initialisation, insertion of admitted keys with their
// rows, and a standalone lookup (MultiTowerDIN: integrating DynamicEmb,
// sections 1 and 3.2). The forward kernel probes the same table inline; see
// hash.cuh for the layout and the probe.
#include <cuda_runtime.h>

#include <cstdint>

#include "dinsparse.h"
#include "hash.cuh"

namespace dsf {
namespace hash {
namespace {

int elem_bytes(int32_t dtype) { return dtype == DSF_BF16 ? 2 : 4; }

bool aligned(const void* q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) & (a - 1)) == 0; }

// Host checks shared by every entry point; fills L.
int check(const dsf_hash* h, Layout& L) {
  if (!h) return DSF_EINVAL;
  if (h->D != 16 && h->D != 64) return DSF_EUNSUPPORTED;
  if (h->dtype != DSF_F32 && h->dtype != DSF_BF16) return DSF_EUNSUPPORTED;
  if (h->capacity < 1 || h->capacity > (1ll << 40)) return DSF_EINVAL;
  L = layout(h->capacity, h->D, elem_bytes(h->dtype));
  if (!h->workspace || !aligned(h->workspace, 256) || h->ws_bytes < L.total) return DSF_EWORKSPACE;
  return DSF_OK;
}

__global__ void init_kernel(uint8_t* ws, Layout L, int D, int dtype, size_t row_bytes) {
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(ws + L.keys_off);
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < (long long)L.n_slots; i += stride)
    keys[i] = kEmptyKey;
  uint32_t* zero = reinterpret_cast<uint32_t*>(ws + L.pool_off + L.n_slots * row_bytes);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < (long long)(row_bytes / 4); i += stride)
    zero[i] = 0u;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    Header* hd = reinterpret_cast<Header*>(ws);
    hd->D = uint32_t(D);
    hd->dtype = uint32_t(dtype);
    hd->pad = 0u;
    hd->n_slots = L.n_slots;
    hd->tag = kHashTag;
  }
}

// One thread per key: claim the key's slot (or find it already present) with
// a compare-and-swap on the first free slot of its probe sequence, then copy
// its row. Every probe is bounded by the bucket count; a key that finds no
// slot sets DSF_FLAG_HASH_FULL and is left out.
__global__ void insert_kernel(uint8_t* ws, Layout L, unsigned int key_space, const long long* __restrict__ raw,
                              const uint8_t* __restrict__ rows, long long n, size_t row_bytes, int* status) {
  const Header* hd = reinterpret_cast<const Header*>(ws);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(ws + L.keys_off);
  uint8_t* pool = ws + L.pool_off;
  int flags = 0;
  const bool ready = hd->tag == kHashTag && hd->n_slots == L.n_slots;
  if (!ready) flags |= DSF_FLAG_HASH;
  const unsigned long long mask = L.n_buckets - 1;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; ready && i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = raw[i];
    if (r < 0 || r >= kKeyLimit) {
      flags |= DSF_FLAG_ID_RANGE;
      continue;
    }
    const unsigned long long k = make_key(key_space, r);
    unsigned long long b = mix64(k) & mask;
    long long slot = -1;
    for (unsigned long long t = 0; t <= mask && slot < 0; ++t, b = (b + 1) & mask) {
      for (int j = 0; j < 8; ++j) {
        unsigned long long* s = keys + (b << 3) + j;
        unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(s);
        if (cur == kEmptyKey) cur = atomicCAS(s, kEmptyKey, k);
        if (cur == kEmptyKey || cur == k) {
          slot = static_cast<long long>((b << 3) + j);
          break;
        }
      }
    }
    if (slot < 0) {
      flags |= DSF_FLAG_HASH_FULL;
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(rows + i * row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(pool + slot * row_bytes);
    for (size_t q = 0; q < row_bytes / 16; ++q) dst[q] = src[q];
  }
  if (flags && status) atomicOr(status, flags);
}

__global__ void find_kernel(const uint8_t* ws, Layout L, unsigned int key_space, const long long* __restrict__ raw,
                            long long n, long long* __restrict__ slot, int* status) {
  const Header* hd = reinterpret_cast<const Header*>(ws);
  const unsigned long long* keys = reinterpret_cast<const unsigned long long*>(ws + L.keys_off);
  const bool ready = hd->tag == kHashTag && hd->n_slots == L.n_slots;
  int flags = ready ? 0 : DSF_FLAG_HASH;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long s = ready ? find(keys, L.n_buckets - 1, key_space, raw[i]) : (long long)L.n_slots;
    if (s == kBadKey) flags |= DSF_FLAG_ID_RANGE;
    slot[i] = s;
  }
  if (flags && status) atomicOr(status, flags);
}

int grid_for(long long n) {
  long long g = (n + 255) / 256;
  if (g < 1) g = 1;
  if (g > 4096) g = 4096;
  return int(g);
}

}  // namespace
}  // namespace hash
}  // namespace dsf

using namespace dsf::hash;

extern "C" size_t dsf_hash_workspace_bytes(int64_t capacity, int32_t D, int32_t dtype) {
  if (capacity < 1 || capacity > (1ll << 40)) return 0;
  if ((D != 16 && D != 64) || (dtype != DSF_F32 && dtype != DSF_BF16)) return 0;
  return layout(capacity, D, elem_bytes(dtype)).total;
}

extern "C" int dsf_hash_init(const dsf_hash* h, void* stream) {
  Layout L;
  const int rc = check(h, L);
  if (rc != DSF_OK) return rc;
  const size_t row_bytes = size_t(h->D) * elem_bytes(h->dtype);
  init_kernel<<<grid_for((long long)L.n_slots), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t*>(h->workspace), L, h->D, h->dtype, row_bytes);
  return cudaGetLastError() == cudaSuccess ? DSF_OK : DSF_ECUDA;
}

extern "C" int dsf_hash_insert(const dsf_hash* h, int32_t key_space, const int64_t* keys_dev, const void* rows_dev,
                               int64_t n, int32_t* status_dev, void* stream) {
  Layout L;
  const int rc = check(h, L);
  if (rc != DSF_OK) return rc;
  if (key_space < 0 || key_space > kMaxKeySpace || n < 0) return DSF_EINVAL;
  if (n == 0) return DSF_OK;
  if (!keys_dev || !rows_dev || !aligned(keys_dev, 8) || !aligned(rows_dev, 16)) return DSF_EINVAL;
  const size_t row_bytes = size_t(h->D) * elem_bytes(h->dtype);
  insert_kernel<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t*>(h->workspace), L, unsigned(key_space), reinterpret_cast<const long long*>(keys_dev),
      static_cast<const uint8_t*>(rows_dev), n, row_bytes, status_dev);
  return cudaGetLastError() == cudaSuccess ? DSF_OK : DSF_ECUDA;
}

extern "C" int dsf_hash_find(const dsf_hash* h, int32_t key_space, const int64_t* keys_dev, int64_t n,
                             int64_t* slots_dev, int32_t* status_dev, void* stream) {
  Layout L;
  const int rc = check(h, L);
  if (rc != DSF_OK) return rc;
  if (key_space < 0 || key_space > kMaxKeySpace || n < 0) return DSF_EINVAL;
  if (n == 0) return DSF_OK;
  if (!keys_dev || !slots_dev || !aligned(keys_dev, 8) || !aligned(slots_dev, 8)) return DSF_EINVAL;
  find_kernel<<<grid_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t*>(h->workspace), L, unsigned(key_space), reinterpret_cast<const long long*>(keys_dev),
      n, reinterpret_cast<long long*>(slots_dev), status_dev);
  return cudaGetLastError() == cudaSuccess ? DSF_OK : DSF_ECUDA;
}
