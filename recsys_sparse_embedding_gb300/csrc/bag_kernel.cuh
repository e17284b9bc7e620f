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
// common case) goes straight through the stage: one thread per bag works out
// the row and output addresses, then each lane group copies rows into its own
// stage slots and stores them from there, two batches of rows and the next
// batch's ids in flight. Bags are summed in value order from zero, as the
// fused kernel and the oracle do, so the results are identical.
#pragma once
#include <cstdint>

#include "fwd_kernel.cuh"

namespace dsf {
namespace bag {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 1024;        // bags per chunk (offsets staged in shared memory)
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
  alignas(16) uint8_t stage[2][kStageBytes / 2];  // two windows' (batches') rows
  union {
    struct {
      long long ids[C::CV];  // the window being issued
      uint8_t feat[C::CV];
    } win;
    struct {
      const uint8_t* src[3][kThreads];  // a batch's row addresses (null: zero row)
      float* dst[3][kThreads];          // its output rows (null: no bag)
    } cp;
  } u;
  long long offs[kChunk + 1];
  long long red[kWarps];
  long long scan[kWarps];
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
  // eight loads in flight per thread per round
  for (long long g = g0 + threadIdx.x; g < g1; g += 8 * kThreads) {
    int v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const long long gk = g + (long long)k * kThreads;
      v[k] = gk < g1 ? __ldg(p.lengths + gk) : 0;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      int x = v[k];
      if (x < 0) { flags |= DSF_FLAG_NEG_LENGTH; x = 0; }
      if (x > kMaxBagLen) { flags |= DSF_FLAG_COUNT; x = kMaxBagLen; }
      tot += x;
    }
  }
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
      // PB bags (as many as half the stage holds, at most one per thread).
      // For batch j, thread t < PB works out bag t's row
      // address and output address (its id loaded one batch ahead) into a
      // ring of three metadata slots; after a barrier, lane group gi copies
      // rows gi, gi + NG, ... of the batch into its stage slots (cp.async),
      // and later stores those same rows from there, so the copies need no
      // further barrier. While batch j is stored, the rows of batch j + 1 and
      // the ids of batch j + 2 are in flight.
      constexpr int PB = (kStageBytes / 2) / C::ROWB < kThreads ? (kStageBytes / 2) / C::ROWB : kThreads;
      constexpr int RB = PB / C::NG;  // rows per lane group per batch
      static_assert(RB >= 1 && RB * C::NG == PB, "a batch is a whole number of rows per lane group");
      const long long vb = sm.offs[0];
      const bool in_range = vb + n <= p.n_values;  // (else per-bag checks below)
      const int nbatch = (n + PB - 1) / PB;
      // bag tid + j * PB: (feature, sample) at the metadata step (fr, br) and
      // at the L2-prefetch step one batch later (fp, bp), advanced by PB per batch
      int fr, br;
      {
        const unsigned x = unsigned(b0) + unsigned(tid);
        fr = f0 + int(x / unsigned(B));
        br = int(x % unsigned(B));
      }
      int fp = fr, bp = br;
      auto load_id = [&](int j) -> long long {
        const int i = j * PB + tid;
        long long id = -1;
        if (tid < PB && i < n && (in_range || vb + i < p.n_values)) id = __ldg(p.values + vb + i);
        return id;
      };
      // bring the row of batch j's bag tid into L2 (plain tables only), two
      // batches before its copy is issued, so that the copy sees L2 latency
      auto prefetch = [&](int j, long long id) {
        if (tid >= PB) return;
        const int i = j * PB + tid;
        if (i < n && !((p.hash_mask >> fp) & 1u) && id >= 0 && id < p.rows[fp])
          prefetch_l2(static_cast<const uint8_t*>(p.tables[fp]) + id * C::ROWB);
        bp += PB;
        while (bp >= B) { bp -= int(B); ++fp; }
      };
      long long idn = -1;
      auto meta = [&](int j) {
        if (tid >= PB) return;
        const int i = j * PB + tid;
        const int m = j % 3;
        const uint8_t* src = nullptr;
        float* dst = nullptr;
        if (i < n) {
          if (in_range || vb + i < p.n_values) {
            long long v = idn;
            if ((p.hash_mask >> fr) & 1u) v = hash::find(p.hkeys, p.hbmask, p.kspace[fr], v);
            if (v >= 0 && v < p.rows[fr]) src = static_cast<const uint8_t*>(p.tables[fr]) + v * C::ROWB;
            else flags |= DSF_FLAG_ID_RANGE;
          } else {
            flags |= DSF_FLAG_COUNT;
          }
          dst = p.pooled + (long long)br * (F * C::D) + fr * C::D;
        }
        sm.u.cp.src[m][tid] = src;
        sm.u.cp.dst[m][tid] = dst;
        br += PB;
        while (br >= B) { br -= int(B); ++fr; }
      };
      // (all of a step's shared-memory loads first, so that their latencies
      // overlap; rows past the chunk have a null output address)
      auto issue = [&](int j) {
        uint8_t* st = sm.stage[j & 1];
        const int m = j % 3;
        const uint8_t* src[RB];
        bool live[RB];
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          const int r = u * C::NG + gi;
          src[u] = sm.u.cp.src[m][r];
          live[u] = sm.u.cp.dst[m][r] != nullptr;
        }
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          const int r = u * C::NG + gi;
          if (live[u])
            cp_async_16_ca(st + r * C::ROWB + sub * 16, src[u] ? src[u] + sub * 16 : p.tables[0], src[u] ? 16u : 0u);
        }
        cp_async_commit();
      };
      auto store = [&](int j) {
        const uint8_t* st = sm.stage[j & 1];
        const int m = j % 3;
        float* o[RB];
        uint4 v[RB];
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          const int r = u * C::NG + gi;
          o[u] = sm.u.cp.dst[m][r];
          v[u] = *reinterpret_cast<const uint4*>(st + r * C::ROWB + sub * 16);
        }
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          if (o[u] != nullptr) {
            float x[C::EPL];
            widen16v<C::BF16>(v[u], x);
            float* q = o[u] + sub * C::EPL;
#pragma unroll
            for (int e = 0; e < C::EPL; e += 4)
              *reinterpret_cast<float4*>(q + e) = make_float4(0.f + x[e], 0.f + x[e + 1], 0.f + x[e + 2], 0.f + x[e + 3]);
          }
        }
      };
      // ids of batches j + 1 (ida) and j + 2 (idb) at the top of step j
      idn = load_id(0);
      long long ida = load_id(1), idb = load_id(2);
      prefetch(0, idn);
      prefetch(1, ida);
      meta(0);
      __syncthreads();
      issue(0);
      for (int j = 0; j < nbatch; ++j) {
        if (j + 2 < nbatch) prefetch(j + 2, idb);
        const long long idc = load_id(j + 3);
        if (j + 1 < nbatch) {
          idn = ida;
          meta(j + 1);   // slot (j + 1) % 3: not read by anyone now
          __syncthreads();
          issue(j + 1);
          cp_async_wait_one_pending();
        } else {
          cp_async_wait_all();
        }
        store(j);
        ida = idb;
        idb = idc;
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
        if (q < nv) sm.u.win.ids[q] = idr[j];
      }
      for (int i = i0 + tid; i < i1 && nv > 0; i += kThreads) {
        int f;
        long long b;
        bag_fb(i, f, b);
        const long long ve = min(sm.offs[i + 1], vs + nv);
        for (long long q = sm.offs[i]; q < ve; ++q) sm.u.win.feat[q - vs] = uint8_t(f);
      }
    };
    // every row copy of a window goes out (one cp.async group)
    auto issue_rows = [&](int i0, int i1, int st) {
      const int nv = nvals(i0, i1);
      for (int q = gi; q < nv; q += C::NG) {
        const int f = sm.u.win.feat[q];
        long long id = sm.u.win.ids[q];
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
