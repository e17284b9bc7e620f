// Hash-table embedding storage (MultiTowerDIN: integrating DynamicEmb,
// sections 1 and 3.2): several large tables share one open-addressing hash
// table and one row pool ("table fusion": shared storage, independent key
// spaces), a raw id is looked up as a key in its table's key space, and a key
// the table does not hold reads the constant zero vector.
//
// Layout of the workspace (caller-owned, 256-byte aligned):
//   [0, 256)           header: tag, D, dtype, slot count
//   [256, 256 + 8 S)   keys, u64 [S]: S = 8 * n_buckets slots in buckets of 8
//                      (one 64-byte line per bucket); kEmptyKey marks a free slot
//   [pool_off, ...)    rows [S + 1][D]: row s belongs to slot s; row S is the
//                      zero row that every unseen key reads
// A stored key is (key_space << 56) | raw, raw in [0, 2^56). Lookups probe
// buckets linearly from the key's hash; a bucket with a free slot ends the
// probe (keys are only ever inserted, never removed).
#pragma once
#include <cstddef>
#include <cstdint>

namespace dsf {
namespace hash {

constexpr unsigned long long kEmptyKey = ~0ull;
constexpr int kKeyBits = 56;
constexpr long long kKeyLimit = 1ll << kKeyBits;
constexpr int kMaxKeySpace = 254;          // key space 255 could form kEmptyKey
constexpr uint32_t kHashTag = 0x48534854u;  // 'THSH'
constexpr long long kBadKey = -2;          // a raw id outside [0, 2^56)

struct Header {
  uint32_t tag, D, dtype, pad;
  unsigned long long n_slots;
};

struct Layout {
  unsigned long long n_buckets, n_slots;
  size_t keys_off, pool_off, total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// capacity: the minimum number of slots; rounded up to 8 * a power of two.
__host__ __device__ inline Layout layout(long long capacity, int D, int elem_bytes) {
  Layout L{};
  unsigned long long nb = 1;
  const unsigned long long want = capacity <= 8 ? 1ull : (unsigned long long)(capacity + 7) / 8;
  while (nb < want) nb <<= 1;
  L.n_buckets = nb;
  L.n_slots = nb * 8;
  L.keys_off = 256;
  L.pool_off = align256(L.keys_off + 8 * L.n_slots);
  L.total = align256(L.pool_off + (L.n_slots + 1) * size_t(D) * size_t(elem_bytes));
  return L;
}

// The finalizer of SplitMix64 (Steele, Lea and Flood, "Fast splittable
// pseudorandom number generators", OOPSLA 2014, with the multipliers of its
// public-domain reference implementation by S. Vigna): a bijective mix of all
// 64 bits, so nearby keys spread over the buckets.
__host__ __device__ __forceinline__ unsigned long long mix64(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

__host__ __device__ __forceinline__ unsigned long long make_key(unsigned int key_space, long long raw) {
  return (static_cast<unsigned long long>(key_space) << kKeyBits) | static_cast<unsigned long long>(raw);
}

// The slot holding `raw` in `key_space`, the zero row's index (n_slots) when
// the table does not hold it, or kBadKey for a raw id outside [0, 2^56). At
// most n_buckets buckets are probed; keys are read through the read-only path
// (no insert runs during a lookup launch).
__device__ __forceinline__ long long find(const unsigned long long* __restrict__ keys, unsigned long long bucket_mask,
                                          unsigned int key_space, long long raw) {
  if (raw < 0 || raw >= kKeyLimit) return kBadKey;
  const unsigned long long k = make_key(key_space, raw);
  unsigned long long b = mix64(k) & bucket_mask;
  for (unsigned long long n = 0; n <= bucket_mask; ++n) {
    const ulonglong2* q = reinterpret_cast<const ulonglong2*>(keys + (b << 3));
    const ulonglong2 w0 = __ldg(q), w1 = __ldg(q + 1), w2 = __ldg(q + 2), w3 = __ldg(q + 3);
    const unsigned long long s[8] = {w0.x, w0.y, w1.x, w1.y, w2.x, w2.y, w3.x, w3.y};
    bool free_slot = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (s[j] == k) return static_cast<long long>((b << 3) + j);
      free_slot |= s[j] == kEmptyKey;
    }
    if (free_slot) break;
    b = (b + 1) & bucket_mask;
  }
  return static_cast<long long>((bucket_mask + 1) << 3);
}

}  // namespace hash
}  // namespace dsf
