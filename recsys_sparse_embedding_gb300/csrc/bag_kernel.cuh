// EmbeddingBag pooling on its own (rows a1-a2 without the attention): the
// pooled rows of every bag of a KJT, for emb_bag_pool and
// emb_bag_pool_noalloc.
//
// MultiTowerDIN: current state analysis, section 3 (the EmbeddingBag layer):
// pooled[b, f] = sum (or mean) of the rows of table f named by bag (f, b).
//
// Two launches. The F*B bags, in the KJT's key-major order, are cut into G
// equal ranges, one per CTA of both; a range's values are one contiguous run
// of the values array, starting at the sum of the lengths of all earlier bags.
// bag_totals_kernel writes each range's length total. bag_kernel then adds up
// the totals of the ranges before its own (plain parallel loads: the first
// launch has finished) and walks its bags in chunks: the chunk's lengths are
// scanned into value offsets in shared memory, and the chunk is cut into
// windows of whole bags holding at most half the row stage. Per window: its
// ids come in with coalesced loads, and every row of the window is copied into
// shared memory at once (cp.async, a group of ROWB/16 lanes per row, so one
// warp instruction touches 32 / (ROWB/16) rows, with hash probes and range
// checks on the way); while window k is summed, one bag per lane group, from
// shared memory, the rows of window k+1 and the ids of window k+2 are in
// flight. A chunk whose bags all hold one value (one id per feature, the
// common case) goes straight through the stage: each lane group copies its
// bags' rows into its own slots and stores them from there, two batches of
// rows and the next batch's ids in flight. Bags are summed in value order from zero, as the
// fused kernel and the oracle do, so the results are identical.
#pragma once
#include <cstdint>

#include "fwd_kernel.cuh"

namespace dsf {
namespace bag {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 2048;        // bags per chunk (offsets staged in shared memory)
constexpr int kStageBytes = 32768;  // row stage: two windows' rows
constexpr long long kMaxWords = (long long)(kWsPartBytes / 8);  // range totals the workspace holds

template <int D_, bool BF16_>
struct Cfg {
  static constexpr int D = D_;
  static constexpr bool BF16 = BF16_;
  static constexpr int ES = BF16 ? 2 : 4;
  static constexpr int ROWB = D * ES;    // bytes per table row
  static constexpr int LPR = ROWB / 16;  // lanes per row
  static constexpr int EPL = 16 / ES;    // elements per lane
  static constexpr int NG = kThreads / LPR;         // row groups per CTA
  static constexpr int CV = kStageBytes / 2 / ROWB;  // values (rows) per window
  static_assert(LPR >= 1 && LPR <= 32 && (32 % LPR) == 0, "a row is a whole number of lanes of one warp");
};

template <class C>
struct Smem {
  alignas(16) uint8_t stage[2][kStageBytes / 2];  // two windows' rows, in value order
  long long ids[C::CV];                           // the window being issued
  long long offs[kChunk + 1];
  long long red[kWarps];
  long long scan[kWarps];
  uint8_t feat[C::CV];
  int flags;
};

__device__ __forceinline__ long long block_sum(long long v, long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  long long s = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) s += red[w];
  return s;
}

// A bag's length as the pooling uses it: negative counts as zero, longer than
// kMaxBagLen is cut there (both flagged).
__device__ __forceinline__ long long bag_len(const FwdParams& p, long long g, int& flags) {
  int v = __ldg(p.lengths + g);
  if (v < 0) { flags |= DSF_FLAG_NEG_LENGTH; v = 0; }
  if (v > kMaxBagLen) { flags |= DSF_FLAG_COUNT; v = kMaxBagLen; }
  return v;
}

__device__ __forceinline__ void report(const FwdParams& p, int flags, int* sm_flags) {
  flags = __reduce_or_sync(0xffffffffu, flags);
  if ((threadIdx.x & 31) == 0 && flags) atomicOr(sm_flags, flags);
  __syncthreads();
  if (threadIdx.x == 0 && *sm_flags) flag(p.status, *sm_flags);
}

// The length total of every CTA's range of bags.
__global__ void __launch_bounds__(kThreads) bag_totals_kernel(const __grid_constant__ FwdParams p) {
  __shared__ long long red[kWarps];
  __shared__ int sm_flags;
  const long long G = gridDim.x, c = blockIdx.x;
  const long long NB = (long long)p.F * p.B;
  const long long g0 = NB * c / G, g1 = NB * (c + 1) / G;
  if (threadIdx.x == 0) sm_flags = 0;
  int flags = 0;
  long long tot = 0;
  for (long long g = g0 + threadIdx.x; g < g1; g += kThreads) tot += bag_len(p, g, flags);
  tot = block_sum(tot, red);
  if (threadIdx.x == 0) p.partials[c] = static_cast<unsigned long long>(tot);
  report(p, flags, &sm_flags);
}

template <class C>
__global__ void __launch_bounds__(kThreads, 4) bag_kernel(const __grid_constant__ FwdParams p) {
  __shared__ Smem<C> sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long G = gridDim.x, c = blockIdx.x;
  const int F = p.F;
  const long long B = p.B, NB = (long long)F * B;
  const long long g0 = NB * c / G, g1 = NB * (c + 1) / G;
  int flags = 0;
  if (tid == 0) sm.flags = 0;
  if (p.hkeys && c == 0 && tid == 0 &&
      (p.hhdr->tag != hash::kHashTag || p.hhdr->n_slots != p.hslots || p.hhdr->D != uint32_t(C::D)))
    flags |= DSF_FLAG_HASH;
  // ---- where this range's values start: the totals of the ranges before it
  long long pre = 0;
  for (long long k = tid; k < c; k += kThreads) pre += static_cast<long long>(p.partials[k]);
  pre = block_sum(pre, sm.red);
  if (c == G - 1 && tid == 0 && pre + static_cast<long long>(p.partials[c]) != p.n_values)
    flags |= DSF_FLAG_COUNT;

  const int gi = tid / C::LPR, sub = tid % C::LPR;  // lane group, 16-byte piece
  long long base = pre;
  bool all_ones = false;
  for (long long cg = g0; cg < g1; cg += kChunk) {
    const int n = int(min((long long)kChunk, g1 - cg));
    // ---- exclusive scan of the chunk's lengths into absolute value offsets
    {
      constexpr int PER = (kChunk + kThreads - 1) / kThreads;
      long long v[PER];
      long long s = 0;
      bool ones = true;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int i = tid * PER + j;
        v[j] = i < n ? bag_len(p, cg + i, flags) : 0;
        ones = ones && (i >= n || v[j] == 1);
        s += v[j];
      }
      all_ones = __syncthreads_and(ones) != 0;
      const long long x = warp_incl_scan(s);
      __syncthreads();
      if (lane == 31) sm.scan[warp] = x;
      __syncthreads();
      long long wpre = 0;
      for (int w = 0; w < warp; ++w) wpre += sm.scan[w];
      long long run = base + wpre + x - s;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int i = tid * PER + j;
        if (i < n) sm.offs[i] = run;
        run += v[j];
      }
      if (tid == kThreads - 1) sm.offs[n] = run;
      __syncthreads();
      base = sm.offs[n];
    }
    const int f0 = int(cg / B), b0 = int(cg - (long long)f0 * B);
    if (all_ones) {
      // Every bag of the chunk holds one value: bag i is value vb + i, and its
      // pooled row is that row (a sum of one; a mean over one). Batches of
      // RB * NG bags; in batch j, lane group gi owns bags j * RB * NG + u * NG
      // + gi (u < RB) and stage slots u * NG + gi of half j % 2: it copies
      // their rows into its slots (cp.async) and later stores them from there,
      // so no barrier is needed. While batch j is stored, the rows of batch
      // j + 1 and the ids of batch j + 2 are in flight. (f, b) of each slot
      // advance by one batch per step.
      constexpr int RB = (kStageBytes / 2) / (C::NG * C::ROWB);
      constexpr int PB = RB * C::NG;  // bags per batch
      const long long vb = sm.offs[0];
      const int nbatch = (n + PB - 1) / PB;
      long long idn[RB];
      int fi[RB], bi[RB], fs[RB], bs_[RB];  // (feature, sample) of the slots at issue / at store
#pragma unroll
      for (int u = 0; u < RB; ++u) {
        const unsigned x = unsigned(b0) + unsigned(u * C::NG + gi);
        fi[u] = fs[u] = f0 + int(x / unsigned(B));
        bi[u] = bs_[u] = int(x % unsigned(B));
      }
      auto advance = [&](int* f, int* b) {
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          b[u] += PB;
          while (b[u] >= B) { b[u] -= int(B); ++f[u]; }
        }
      };
      auto load_ids = [&](int j) {
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          const int i = j * PB + u * C::NG + gi;
          idn[u] = -1;
          if (i < n) {
            if (vb + i < p.n_values) idn[u] = __ldg(p.values + vb + i);
            else if (sub == 0) flags |= DSF_FLAG_COUNT;
          }
        }
      };
      auto issue = [&](int j) {
        uint8_t* st = sm.stage[j & 1];
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          const int i = j * PB + u * C::NG + gi;
          if (i < n) {
            long long v = idn[u];
            const int f = fi[u];
            bool ok = false;
            if (vb + i < p.n_values) {
              if ((p.hash_mask >> f) & 1u) v = hash::find(p.hkeys, p.hbmask, p.kspace[f], v);
              ok = v >= 0 && v < p.rows[f];
              if (!ok && sub == 0) flags |= DSF_FLAG_ID_RANGE;
            }
            const uint8_t* src = static_cast<const uint8_t*>(p.tables[f]) + (ok ? v : 0) * C::ROWB + sub * 16;
            cp_async_16_ca(st + (u * C::NG + gi) * C::ROWB + sub * 16, src, ok ? 16u : 0u);
          }
        }
        cp_async_commit();
        advance(fi, bi);
      };
      auto store = [&](int j) {
        const uint8_t* st = sm.stage[j & 1];
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          const int i = j * PB + u * C::NG + gi;
          if (i < n) {
            float x[C::EPL];
            widen16<C::BF16>(st + (u * C::NG + gi) * C::ROWB + sub * 16, x);
            float* o = p.pooled + (long long)bs_[u] * (F * C::D) + fs[u] * C::D + sub * C::EPL;
#pragma unroll
            for (int e = 0; e < C::EPL; e += 4)
              *reinterpret_cast<float4*>(o + e) = make_float4(0.f + x[e], 0.f + x[e + 1], 0.f + x[e + 2], 0.f + x[e + 3]);
          }
        }
        advance(fs, bs_);
      };
      load_ids(0);
      issue(0);
      if (nbatch > 1) load_ids(1);
      for (int j = 0; j < nbatch; ++j) {
        if (j + 1 < nbatch) issue(j + 1);
        if (j + 2 < nbatch) load_ids(j + 2);
        if (j + 1 < nbatch) cp_async_wait_one_pending();
        else cp_async_wait_all();
        store(j);
      }
      __syncthreads();  // before the next chunk's offsets
      continue;
    }
    // bag i of the chunk is bag (f0 + (b0 + i) / B, (b0 + i) % B): 32-bit
    // division (b0 < B < 2^25, i < kChunk)
    const unsigned UB = unsigned(B);
    auto bag_fb = [&](int i, int& f, long long& b) {
      const unsigned x = unsigned(b0) + unsigned(i), q = x / UB;
      f = f0 + int(q);
      b = (long long)(x - q * UB);
    };
    // ---- windows: bags [i0, i1) with at most CV values (at least one bag; a
    // bag longer than that is summed straight from global memory)
    auto window_end = [&](int i0) -> int {
      return min(n, max(i0 + 1, upper_index(sm.offs + i0, n - i0 + 1, sm.offs[i0] + C::CV) + i0));
    };
    auto nvals = [&](int i0, int i1) -> int {  // staged values of a window (0: not staged)
      const long long vs = sm.offs[i0];
      if (sm.offs[i1] - vs > C::CV) return 0;
      return int(max(0ll, min(sm.offs[i1], p.n_values) - vs));
    };
    // a window's ids: loads into registers (in flight while the CTA works),
    // then into shared memory with the feature of each value
    constexpr int IPT = (C::CV + kThreads - 1) / kThreads;
    long long idr[IPT];
    auto load_ids = [&](int i0, int i1) {
      const long long vs = sm.offs[i0];
      const int nv = nvals(i0, i1);
#pragma unroll
      for (int j = 0; j < IPT; ++j) {
        const int q = tid + j * kThreads;
        idr[j] = q < nv ? __ldg(p.values + vs + q) : 0;
      }
    };
    auto store_ids = [&](int i0, int i1) {
      const long long vs = sm.offs[i0];
      const int nv = nvals(i0, i1);
#pragma unroll
      for (int j = 0; j < IPT; ++j) {
        const int q = tid + j * kThreads;
        if (q < nv) sm.ids[q] = idr[j];
      }
      for (int i = i0 + tid; i < i1 && nv > 0; i += kThreads) {
        int f;
        long long b;
        bag_fb(i, f, b);
        const long long ve = min(sm.offs[i + 1], vs + nv);
        for (long long q = sm.offs[i]; q < ve; ++q) sm.feat[q - vs] = uint8_t(f);
      }
    };
    // every row copy of a window goes out (one cp.async group)
    auto issue_rows = [&](int i0, int i1, int st) {
      const int nv = nvals(i0, i1);
      for (int q = gi; q < nv; q += C::NG) {
        const int f = sm.feat[q];
        long long id = sm.ids[q];
        if ((p.hash_mask >> f) & 1u) id = hash::find(p.hkeys, p.hbmask, p.kspace[f], id);
        const bool ok = id >= 0 && id < p.rows[f];
        if (!ok && sub == 0) flags |= DSF_FLAG_ID_RANGE;
        const uint8_t* src = static_cast<const uint8_t*>(p.tables[f]) + (ok ? id : 0) * C::ROWB + sub * 16;
        cp_async_16_ca(sm.stage[st] + q * C::ROWB + sub * 16, src, ok ? 16u : 0u);
      }
      cp_async_commit();
    };
    // the sums, one bag per lane group, in value order from zero
    auto sum = [&](int i0, int i1, int st) {
      const long long vs = sm.offs[i0];
      const bool staged = sm.offs[i1] - vs <= C::CV;
      for (int i = i0 + gi; i < i1; i += C::NG) {
        int f;
        long long b;
        bag_fb(i, f, b);
        const long long va = sm.offs[i];
        long long ve = sm.offs[i + 1];
        if (ve > p.n_values) { flags |= DSF_FLAG_COUNT; ve = va; }
        float acc[C::EPL];
#pragma unroll
        for (int e = 0; e < C::EPL; ++e) acc[e] = 0.f;
        if (staged) {
          for (long long q = va; q < ve; ++q) {
            float x[C::EPL];
            widen16<C::BF16>(sm.stage[st] + (q - vs) * C::ROWB + sub * 16, x);
#pragma unroll
            for (int e = 0; e < C::EPL; ++e) acc[e] += x[e];
          }
        } else {
          for (long long q = va; q < ve; ++q) {
            long long v = __ldg(p.values + q);
            if ((p.hash_mask >> f) & 1u) v = hash::find(p.hkeys, p.hbmask, p.kspace[f], v);
            if (v < 0 || v >= p.rows[f]) { if (sub == 0) flags |= DSF_FLAG_ID_RANGE; continue; }
            float x[C::EPL];
            widen16v<C::BF16>(ldg16(static_cast<const uint8_t*>(p.tables[f]) + v * C::ROWB + sub * 16), x);
#pragma unroll
            for (int e = 0; e < C::EPL; ++e) acc[e] += x[e];
          }
        }
        if ((p.mean_mask >> f) & 1u) {
          // mean pooling: the fp32 sum over the bag's length (empty stays 0)
          const long long L = sm.offs[i + 1] - sm.offs[i];
          if (L > 0) {
#pragma unroll
            for (int e = 0; e < C::EPL; ++e) acc[e] = acc[e] / float(L);
          }
        }
        float* o = p.pooled + b * (F * C::D) + f * C::D + sub * C::EPL;
#pragma unroll
        for (int e = 0; e < C::EPL; e += 4)
          *reinterpret_cast<float4*>(o + e) = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
      }
    };
    // The pipeline, three windows deep: at step k the rows of window k+1 go
    // out, the ids of window k+2 are loaded, window k is summed.
    int w0 = 0, w1 = window_end(0), st = 0;
    load_ids(w0, w1);
    store_ids(w0, w1);
    __syncthreads();
    issue_rows(w0, w1, st);
    int w2 = w1 < n ? window_end(w1) : w1;
    if (w1 < n) {
      __syncthreads();  // (window 0's copies have read the ids)
      load_ids(w1, w2);
      store_ids(w1, w2);
      __syncthreads();
    }
    while (w0 < n) {
      const bool more = w1 < n;
      if (more) issue_rows(w1, w2, st ^ 1);
      const int w3 = w2 < n ? window_end(w2) : w2;
      if (w2 < n) load_ids(w2, w3);
      if (more) cp_async_wait_one_pending();
      else cp_async_wait_all();
      __syncthreads();  // window 0's rows have landed; the ids were read
      sum(w0, w1, st);
      __syncthreads();  // stage st is free again
      if (w2 < n) {
        store_ids(w2, w3);
        __syncthreads();
      }
      w0 = w1;
      w1 = w2;
      w2 = w3;
      st ^= 1;
    }
  }
  report(p, flags, &sm.flags);
}

}  // namespace bag
}  // namespace dsf
