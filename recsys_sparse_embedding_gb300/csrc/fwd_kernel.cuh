// Fused MultiTowerDIN sparse forward for sm_103a: KJT offsets scan, sum-pooled
// EmbeddingBag gather and padding-free DIN target attention in one persistent,
// cooperatively launched kernel (one CTA per SM when attention is on).
//
// Method (pages cited by title and section):
//   "MultiTowerDIN: current state analysis"
//     s2   SparseData(values, lengths) -> KeyedJaggedTensor; sequence features
//          carry (values, seq_lengths)
//     s3   one [num_buckets, 16] table per id feature, sum-pooled bags
//     s4.1 the sequence is padded to 100 in the pages' flow; here only the
//          valid positions are ever gathered or computed
//     s4.2 attention input cat[q, s, q - s, q * s]; attn_mlp 256 -> 64, linear
//          to 1, mask + softmax, weighted sum
//     s4.4 shapes [B,48] query, [B,100,192] input, [B,48] output
//   "MultiTowerDIN: integrating DynamicEmb"
//     s2.4 sequence sub-features share the target features' tables
//     s3.3 lookup in fp32, MLP in half precision (bf16 here)
//
// Work split. CTA c takes the contiguous samples [c*B/G, (c+1)*B/G). It pools
// all F bags of its own samples (so each pooled row is written by one
// CTA) and then runs attention for the same samples, so the query never
// crosses CTAs. The only cross-CTA exchange is the per-feature length total of
// each CTA's samples, needed to place its bags in the key-major values array.
// Each CTA publishes its totals tagged with the launch epoch; a CTA that needs
// them polls the tagged words themselves (bounded wait), so the exchange costs
// one round trip once the last CTA has published. The first sequence tile's
// gather is in flight meanwhile. The epoch advances when the last CTA exits.
#pragma once
#include <cstdint>
#include <type_traits>

#include "dinsparse.h"
#include "hash.cuh"
#include "ptx.cuh"

namespace dsf {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kSB = 128;            // samples per batch inside a CTA (<= 256: uint8 row metadata)
constexpr int kMaxF = 32;           // tables
constexpr int kMaxG = 1024;         // grid size limit (rows of the partials table)
constexpr int kN1 = 256, kN2 = 64;  // attn_mlp hidden units
constexpr int kMaxBagLen = 1 << 19; // longer bags are clamped (flagged)
constexpr int kShortBag = 16;       // batches whose bags all fit pool directly

// Workspace layout (bytes). The header holds the prepared-weights tag, the
// launch epoch and the exit counter that advances it.
constexpr size_t kWsMagicOff = 0;
constexpr size_t kWsEpochOff = 128;
constexpr size_t kWsPartOff = 256;
constexpr size_t kWsPartBytes = size_t(kMaxG) * kMaxF * 8;
constexpr size_t kWsWpackOff = kWsPartOff + kWsPartBytes;
constexpr uint32_t kMagicBase = 0x44534600u;  // 'DSF\0' | D

struct FwdParams {
  const void* tables[kMaxF];
  long long rows[kMaxF];
  int F, B, max_len;
  unsigned int mean_mask;  // bit f: table f pools by mean
  const long long* values;
  long long n_values;
  const int* lengths;
  const long long* seq_values;
  long long n_seq;
  const int* seq_lengths;
  int q_feat[3], seq_table[3];
  float* pooled;   // [B, F*D] or null
  float* qbuf;     // [B, 3D] query buffer when pooled is null
  float* din;      // [B, 3D] (attention)
  float* logits;   // [n_seq] or null
  const float *b1, *b2, *w3, *b3;
  const uint8_t* wpack;  // bf16 W1 | W2 in the swizzled operand layout
  const float* w1t;      // fp32 W1^T [K1][256]
  const float* w2t;      // fp32 W2^T [256][64]
  const uint32_t* magic;
  // hash-table storage (null hkeys: none): tables in hash_mask read the fused
  // row pool at the slot of their raw key in key space kspace[f]
  const unsigned long long* hkeys;
  const hash::Header* hhdr;
  unsigned long long hbmask;  // buckets - 1
  unsigned long long hslots;  // slots (the zero row's index)
  unsigned int hash_mask;
  unsigned char kspace[kMaxF];
  unsigned int* epoch;           // launch counter, tags the partials
  unsigned long long* partials;  // (epoch + 1) << 32 | length total: [G][kMaxF] here, [G] for pooling alone
  int* status;
};

// ------------------------------------------------------------------ config
template <int D_, bool BF16_, int MODE_, bool ATTN_>
struct Cfg {
  static constexpr int D = D_;
  static constexpr bool BF16 = BF16_;  // table element type
  static constexpr int MODE = MODE_;   // 0: bf16 tcgen05 MLP, 1: fp32 CUDA-core MLP
  static constexpr bool ATTN = ATTN_;
  static constexpr int ES = BF16 ? 2 : 4;
  static constexpr int ROWB = D * ES;          // bytes per table row
  static constexpr int LPB = ROWB / 16;        // 16-byte pieces per row
  static constexpr int EPL = 16 / ES;          // elements per 16-byte piece
  static constexpr int Q = 3 * D;
  static constexpr int K1 = 4 * Q;
  static constexpr int TM = MODE == 0 ? 128 : 64;  // rows per attention tile
  // bytes per S row; the tensor-core mode pads each row by 16 bytes so that a
  // warp reading one 16-byte piece of 32 consecutive rows hits every bank
  static constexpr int SROWB = Q * ES + (MODE == 0 ? 16 : 0);
  static constexpr int QROW = Q + 4;               // floats per q-tile row (padded)
  static_assert(D % 8 == 0, "D must be a multiple of 8");

  // pool region: bag offsets at its end (F*nb+1 words), staging rows before
  static constexpr int POOL_BYTES = 64 * 1024;

  // tensor-core mode
  static constexpr int W1B = kN1 * K1 * 2;
  static constexpr int W2B = kN2 * kN1 * 2;
  static constexpr int XB = TM * K1 * 2;
  static constexpr int H1B = TM * kN1 * 2;
  // fp32 mode
  static constexpr int H1S = kN1 + 4;  // padded fp32 row stride
  static constexpr int QTB = TM * Q * 4;
  static constexpr int H1FB = TM * H1S * 4;

  static constexpr int cmax(int a, int b) { return a > b ? a : b; }

  // Byte offsets from the 1024-aligned smem base. In the tensor-core mode the
  // attention input x and h1 live in tensor memory, and the sequence rows S are
  // double-buffered: [W1 | W2 | ACT | S1 | S0 | misc]. Pooling stages rows in
  // ACT and S1 (S1 is free then: only the first tile is in flight, in S0).
  // With D = 64 the 768-wide W1 does not fit: it streams through a ring of
  // W1_STAGES K-blocks (64 wide, 32 KB) and x is built one K-block at a time in
  // a two-slot smem ring: [W2 | W1 ring | x ring | S | misc]; pooling stages in
  // the W1 and x rings.
  static constexpr bool STREAM = ATTN && MODE == 0 && D == 64;
  static constexpr bool TWO_S = ATTN && MODE == 0 && !STREAM;
  static constexpr int W1_STAGES = 3;
  static constexpr int W1KB = kN1 * 128;     // one 64-wide K-block of W1
  static constexpr int XKB = TM * 128;       // one 64-wide K-block of x
  static constexpr int W1_OFF = STREAM ? W2B : 0;
  static constexpr int W2_OFF = STREAM ? 0 : ((ATTN && MODE == 0) ? W1_OFF + W1B : 0);
  static constexpr int XR_OFF = W1_OFF + W1_STAGES * W1KB;  // stream mode
  static constexpr int ACT_OFF = STREAM ? W1_OFF : ((ATTN && MODE == 0) ? W2_OFF + W2B : 0);
  static constexpr int ACT_BYTES =
      !ATTN ? POOL_BYTES
            : (STREAM ? W1_STAGES * W1KB + 2 * XKB
                      : (MODE == 0 ? (kSB * QROW * 4 + 1023) / 1024 * 1024 : cmax(H1FB, POOL_BYTES)));
  static constexpr int QT_OFF = ACT_OFF + ACT_BYTES;  // fp32 mode only
  static constexpr int S_BYTES = ATTN ? TM * SROWB : 0;
  static constexpr int S1_OFF = QT_OFF + ((ATTN && MODE == 1) ? QTB : 0);
  static constexpr int S_OFF = S1_OFF + (TWO_S ? S_BYTES : 0);  // buffer 0
  // pipelined tiles: the bias operands of the extra K-step of each layer
  // (N rows of 16 bf16: b_hi, b_lo, zeros; 32-byte swizzled K-major)
  static constexpr int BIAS1B = kN1 * 32, BIAS2B = kN2 * 32;
  static constexpr int BIAS_OFF = S_OFF + S_BYTES;
  static constexpr int MISC_OFF = (BIAS_OFF + (TWO_S ? BIAS1B + BIAS2B : 0) + 127) / 128 * 128;
  static constexpr int POOL_AVAIL = ACT_BYTES + (TWO_S ? S_BYTES : 0);
  // values a thread stages per pooling window
  static constexpr int VPT = (POOL_AVAIL / ROWB + kThreads - 1) / kThreads;
  // tensor-memory columns: layer-1 accumulator (h1 packed over its first half),
  // layer-2 accumulator, the bf16 x tile
  static constexpr uint32_t TM_ACC1 = 0, TM_ACC2 = kN1, TM_X = kN1 + kN2;
  // pipelined tiles: 8 constant columns, the A operand of the bias K-step (1, 1, 0 ...)
  static constexpr uint32_t TM_ONE = TM_X + K1 / 2;
  static_assert(!TWO_S || TM_ONE + 8 <= 512, "tensor memory columns");
  static_assert(!TWO_S || kSB * QROW * 4 <= ACT_BYTES, "query slices of a batch");
  static_assert(32 + 3 * TM <= kThreads, "sequence rows: one thread per (row, key) outside warp 0");
};

template <int D, int Q>
struct Misc {
  float b1[kN1];
  float b2[kN2];
  float w3[kN2];
  float z[128];
  float red[4][128];
  float carry[2][4 + Q];       // softmax state: m, l, -, -, acc[Q]
  float pcarry[2][D];          // pooling carry of a bag that spans windows
  uint8_t row_samp[4][128];     // per tile (ring of 4): sample (in the batch) of each row
  int rp[kSB + 4];             // valid-row prefix of the batch's samples
  int so[kSB];                 // first sequence value index of each sample
  long long fcur[kMaxF];       // next global value index of feature f for this CTA
  long long ftb[kMaxF];        // value count of feature f in the current batch
  long long ft[kMaxF];
  long long fpre[kMaxF];
  long long scan64[2][kWarps + 2];
  long long cred[kWarps + 1];   // block_scan2_sum: per-warp sums, then the total
  uint64_t mbar_w;
  uint64_t mbar_mma;
  uint64_t mbar_full[3];       // W1 K-block landed in ring slot (stream mode)
  uint64_t mbar_done[3];       // MMAs reading ring slot finished (stream mode)
  unsigned int tmem_base;
  int abort_;
  long long seq_cur;           // seq value index of the next batch's first sample
  unsigned int epoch;
};

template <class C>
constexpr int smem_bytes() {
  return C::MISC_OFF + int(sizeof(Misc<C::D, C::Q>)) + 1024;  // + alignment slack
}

// ------------------------------------------------------------------ helpers
template <typename T>
__device__ __forceinline__ T warp_incl_scan(T v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Exclusive scan of two int64 values over the block. Contains __syncthreads.
__device__ __forceinline__ void block_scan2(long long a, long long b, long long (*scr)[kWarps + 2],
                                            long long& ea, long long& eb, long long& ta,
                                            long long& tb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long ia = warp_incl_scan(a), ib = warp_incl_scan(b);
  if (lane == 31) {
    scr[0][warp] = ia;
    scr[1][warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    long long wa = lane < kWarps ? scr[0][lane] : 0;
    long long wb = lane < kWarps ? scr[1][lane] : 0;
    long long xa = warp_incl_scan(wa), xb = warp_incl_scan(wb);
    if (lane < kWarps) {
      scr[0][lane] = xa - wa;
      scr[1][lane] = xb - wb;
    }
    if (lane == kWarps - 1) {
      scr[0][kWarps] = xa;
      scr[1][kWarps] = xb;
    }
  }
  __syncthreads();
  ea = scr[0][warp] + ia - a;
  eb = scr[1][warp] + ib - b;
  ta = scr[0][kWarps];
  tb = scr[1][kWarps];
  __syncthreads();
}

// block_scan2 of (a, b) plus the block-wide total of c (cscr: kWarps + 1 words).
__device__ __forceinline__ void block_scan2_sum(long long a, long long b, long long c,
                                                long long (*scr)[kWarps + 2], long long* cscr,
                                                long long& ea, long long& eb, long long& ta,
                                                long long& tb, long long& tc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long ia = warp_incl_scan(a), ib = warp_incl_scan(b), sc = warp_sum(c);
  if (lane == 31) {
    scr[0][warp] = ia;
    scr[1][warp] = ib;
    cscr[warp] = sc;
  }
  __syncthreads();
  if (warp == 0) {
    long long wa = lane < kWarps ? scr[0][lane] : 0;
    long long wb = lane < kWarps ? scr[1][lane] : 0;
    long long wc = lane < kWarps ? cscr[lane] : 0;
    long long xa = warp_incl_scan(wa), xb = warp_incl_scan(wb);
    wc = warp_sum(wc);
    if (lane < kWarps) {
      scr[0][lane] = xa - wa;
      scr[1][lane] = xb - wb;
    }
    if (lane == kWarps - 1) {
      scr[0][kWarps] = xa;
      scr[1][kWarps] = xb;
      cscr[kWarps] = wc;
    }
  }
  __syncthreads();
  ea = scr[0][warp] + ia - a;
  eb = scr[1][warp] + ib - b;
  ta = scr[0][kWarps];
  tb = scr[1][kWarps];
  tc = cscr[kWarps];
  __syncthreads();
}

// Largest i in [0, n) with a[i] <= x (a non-decreasing, a[0] <= x).
template <typename T>
__device__ __forceinline__ int upper_index(const T* a, int n, long long x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if ((long long)a[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void flag(int* status, int bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ float4 ldcg4(const float* p) {
  return __ldcg(reinterpret_cast<const float4*>(p));
}

// 16 bytes of a read-only table row, through the non-coherent path.
__device__ __forceinline__ uint4 ldg16(const uint8_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// 16-byte piece of a row (fp32 or bf16) widened to EPL floats.
template <bool BF16>
__device__ __forceinline__ void widen16v(const uint4 v, float* out) {
  if constexpr (BF16) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[2 * i] = __uint_as_float(w[i] << 16);
      out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
    out[0] = __uint_as_float(v.x);
    out[1] = __uint_as_float(v.y);
    out[2] = __uint_as_float(v.z);
    out[3] = __uint_as_float(v.w);
  }
}

template <bool BF16>
__device__ __forceinline__ void widen16(const uint8_t* src, float* out) {
  widen16v<BF16>(*reinterpret_cast<const uint4*>(src), out);
}

template <bool BF16>
__device__ __forceinline__ float s_elem(const uint8_t* S, int srowb, int r, int d) {
  if constexpr (BF16) {
    const uint16_t h = *reinterpret_cast<const uint16_t*>(S + r * srowb + d * 2);
    return __uint_as_float(uint32_t(h) << 16);
  } else {
    return *reinterpret_cast<const float*>(S + r * srowb + d * 4);
  }
}

// Elements d .. d+3 of row r of a staged S tile (d a multiple of 4).
template <bool BF16>
__device__ __forceinline__ float4 s_quad(const uint8_t* S, int srowb, int r, int d) {
  if constexpr (BF16) {
    const uint2 h = *reinterpret_cast<const uint2*>(S + r * srowb + d * 2);
    return make_float4(__uint_as_float(h.x << 16), __uint_as_float(h.x & 0xffff0000u),
                       __uint_as_float(h.y << 16), __uint_as_float(h.y & 0xffff0000u));
  } else {
    return *reinterpret_cast<const float4*>(S + r * srowb + d * 4);
  }
}

// ------------------------------------------------------------------ kernel
template <class C>
__global__ void __launch_bounds__(kThreads, 1) dsf_fwd_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using M = Misc<C::D, C::Q>;
  M* ms = reinterpret_cast<M*>(sm + C::MISC_OFF);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, cta = blockIdx.x;
  const int F = p.F, B = p.B;
  constexpr int D = C::D, Q = C::Q;
  int local_flags = 0;

  // ---------------------------------------------------------------- partition
  // Equal sample counts per CTA: no cross-CTA work is needed to place them.
  const int sb0 = int((long long)cta * B / G);
  const int sb1 = int((long long)(cta + 1) * B / G);
  const int ns = sb1 - sb0;
  const int nb0 = min(kSB, ns);

  // ---------------------------------------------------------------- early loads
  // Every global read the first phases depend on goes out before the
  // prologue, so that their latencies overlap: the launch epoch and prepared
  // tag, the first batch's bag lengths (pooling scan), its sequence lengths
  // (batch setup) and the first pass of sequence lengths before it (offset).
  const unsigned int epoch = *p.epoch;
  const uint32_t magic = C::ATTN ? *p.magic : 0u;
  // Bag lengths of a batch, one feature per warp: warp w holds features
  // w + kWarps*a (a < kLF), lane l the samples l + 32j (j < kLJ).
  constexpr int kLF = (kMaxF + kWarps - 1) / kWarps, kLJ = kSB / 32;
  int lenv[kLF][kLJ];
  auto pool_len_load = [&](int bs, int nb) {
#pragma unroll
    for (int a = 0; a < kLF; ++a) {
      const int f = warp + a * kWarps;
#pragma unroll
      for (int j = 0; j < kLJ; ++j) {
        const int i = lane + 32 * j;
        lenv[a][j] = (f < F && i < nb) ? p.lengths[(long long)f * B + bs + i] : 0;
      }
    }
  };
  if (ns > 0) pool_len_load(sb0, nb0);
  const int seq_len0 = (C::ATTN && tid < nb0) ? p.seq_lengths[sb0 + tid] : 0;
  int seq_pre[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int b = k * kThreads + tid;
    seq_pre[k] = (C::ATTN && b < sb0) ? p.seq_lengths[b] : 0;
  }

  // ---------------------------------------------------------------- prologue
  // The biases and the weights are copied asynchronously.
  bool attn_ok = C::ATTN;
  if (tid == 0) {
    ms->abort_ = 0;
    if constexpr (C::ATTN && C::MODE == 0) {
      mbar_init(&ms->mbar_w, 1);
      mbar_init(&ms->mbar_mma, 1);
      if constexpr (C::STREAM) {
        for (int i = 0; i < 3; ++i) {
          mbar_init(&ms->mbar_full[i], 1);
          mbar_init(&ms->mbar_done[i], 1);
        }
      }
      fence_mbarrier_init();
      // stage the packed bf16 weights (bulk copies, 16 KB pieces): W1 | W2, or
      // only W2 when W1 streams
      const int w_src = C::STREAM ? C::W1B : 0;
      const int w_bytes = C::STREAM ? C::W2B : C::W1B + C::W2B;
      uint8_t* w_dst = sm + (C::STREAM ? C::W2_OFF : C::W1_OFF);
      mbar_arrive_expect_tx(&ms->mbar_w, w_bytes);
      for (int off = 0; off < w_bytes; off += 16384) {
        const int nbytes = min(16384, w_bytes - off);
        bulk_g2s(w_dst + off, p.wpack + w_src + off, nbytes, &ms->mbar_w);
      }
    }
  }
  if constexpr (C::ATTN) {
    if constexpr (C::MODE == 0) {
      __syncwarp();
      if (warp == 0) {
        tmem_alloc(&ms->tmem_base, 512);
        tmem_relinquish();
        tc_fence_before();
      }
    }
    // biases: 16-byte pieces of b1 [256], b2 [64], w3 [64]
    if (tid < kN1 / 4) cp_async_16_ca(ms->b1 + 4 * tid, p.b1 + 4 * tid, 16u);
    else if (tid < kN1 / 4 + kN2 / 4) cp_async_16_ca(ms->b2 + 4 * (tid - kN1 / 4), p.b2 + 4 * (tid - kN1 / 4), 16u);
    else if (tid < kN1 / 4 + kN2 / 2) cp_async_16_ca(ms->w3 + 4 * (tid - kN1 / 4 - kN2 / 4), p.w3 + 4 * (tid - kN1 / 4 - kN2 / 4), 16u);
  }
  __syncthreads();
  if constexpr (C::ATTN && C::MODE == 0) tc_fence_after();
  const float b3 = C::ATTN ? __ldg(p.b3) : 0.f;

  attn_ok = C::ATTN && magic == (kMagicBase | uint32_t(D));
  if (C::ATTN && tid == 0 && !attn_ok && cta == 0) flag(p.status, DSF_FLAG_NOT_PREPARED);
  // the hash workspace's header, checked once (off the critical threads)
  if (p.hkeys && cta == 0 && tid == kThreads - 1 &&
      (p.hhdr->tag != hash::kHashTag || p.hhdr->n_slots != p.hslots || p.hhdr->D != uint32_t(D)))
    flag(p.status, DSF_FLAG_HASH);
  const unsigned long long tag = (unsigned long long)(epoch + 1u) << 32;

  // ---------------------------------------------------------------- pooling helpers
  // Bag offsets of a batch of nb samples live at the end of the pool region
  // (F*nb+1 words); value rows are staged before them, `cap` rows per window.
  const bool pool_all = p.pooled != nullptr;
  auto want_feature = [&](int f) -> bool {
    if (pool_all) return true;
    return f == p.q_feat[0] || f == p.q_feat[1] || f == p.q_feat[2];
  };
  auto pool_offs = [&](int nb) -> uint32_t* {
    const int offs_bytes = ((F * nb + 1) * 4 + 15) / 16 * 16;
    return reinterpret_cast<uint32_t*>(sm + C::ACT_OFF + C::POOL_AVAIL - offs_bytes);
  };
  auto pool_cap = [&](int nb) -> int {
    const int offs_bytes = ((F * nb + 1) * 4 + 15) / 16 * 16;
    return (C::POOL_AVAIL - offs_bytes) / C::ROWB;
  };
  // bag g -> feature g / nb as a multiply-shift, exact for g < 4097, nb <= 128
  auto nb_recip_of = [](int nb) -> unsigned { return ((1u << 20) + unsigned(nb) - 1u) / unsigned(nb); };
  // Exclusive scan of the batch's bag lengths (key-major bags g = f*nb + i,
  // from pool_len_load) into offs; returns the batch's value count and
  // whether any bag holds more than kShortBag values. With publish, each
  // feature's total is stored to this CTA's partials row as soon as its warp
  // has summed it. Contains barriers.
  auto pool_scan = [&](int nb, bool& longbag, bool publish) -> long long {
    uint32_t* offs = pool_offs(nb);
    bool lng = false;
#pragma unroll
    for (int a = 0; a < kLF; ++a) {
      long long sf = 0;
#pragma unroll
      for (int j = 0; j < kLJ; ++j) {
        int& v = lenv[a][j];
        if (v < 0) { local_flags |= DSF_FLAG_NEG_LENGTH; v = 0; }
        if (v > kMaxBagLen) { local_flags |= DSF_FLAG_COUNT; v = kMaxBagLen; }
        lng = lng || v > kShortBag;
        sf += v;
      }
      sf = warp_sum(sf);
      const int f = warp + a * kWarps;
      if (lane == 0 && f < F) {
        ms->ftb[f] = sf;
        if (publish) {
          if (sf > 0x7fffffffll) { local_flags |= DSF_FLAG_COUNT; sf = 0x7fffffffll; }
          // (each word carries its own tag: no fence needed behind it)
          st_relaxed_u64(&p.partials[(long long)cta * kMaxF + f], tag | (unsigned long long)sf);
        }
      }
    }
    longbag = __syncthreads_or(lng) != 0;
    // feature f starts after all bags of features < f
    const long long tf = lane < F ? ms->ftb[lane] : 0;
    const long long incl = warp_incl_scan(tf);
    const long long tot = __shfl_sync(0xffffffffu, incl, 31);
#pragma unroll
    for (int a = 0; a < kLF; ++a) {
      const int f = warp + a * kWarps;
      if (f >= F) continue;  // warp-uniform
      long long base = __shfl_sync(0xffffffffu, incl - tf, f);
#pragma unroll
      for (int j = 0; j < kLJ; ++j) {
        const long long v = lenv[a][j];
        const long long in = warp_incl_scan(v);
        const int i = lane + 32 * j;
        if (i < nb) offs[f * nb + i] = uint32_t(base + in - v);
        base += __shfl_sync(0xffffffffu, in, 31);
      }
    }
    if (tid == 0) offs[F * nb] = uint32_t(tot);
    __syncthreads();
    return tot;
  };
  // For the values [w0, w1) of a window: bag -> (feature, index within the
  // feature's values of this batch), kept in each value's own staging slot
  // until its id is loaded.
  auto pool_map = [&](int nb, long long w0, long long w1) {
    const uint32_t* offs = pool_offs(nb);
    const unsigned rcp = nb_recip_of(nb);
    for (long long u = w0 + tid; u < w1; u += kThreads) {
      const int g = upper_index(offs, F * nb + 1, u);
      const int f = int((unsigned(g) * rcp) >> 20);
      *reinterpret_cast<int2*>(sm + C::ACT_OFF + (u - w0) * C::ROWB) =
          make_int2(f, int(u - (long long)offs[f * nb]));
    }
  };

  // ---------------------------------------------------------------- per-feature totals
  // The first batch's bag offsets (and its first window's value map) are made
  // here, before the exchange; a CTA with a single batch publishes its totals
  // straight from them.
  long long U0 = 0;
  bool long0 = false;
  if (tid < kMaxF) {
    ms->ft[tid] = 0;
    ms->fpre[tid] = 0;
  }
  if (ns > 0) U0 = pool_scan(nb0, long0, ns <= kSB);
  if (ns == 0) {
    if (tid < F) st_relaxed_u64(&p.partials[(long long)cta * kMaxF + tid], tag);
  } else if (ns > kSB) for (int f = warp; f < F; f += kWarps) {
    long long s = 0;
    const int* lp = p.lengths + (long long)f * B + sb0;
    for (int i0 = 0; i0 < ns; i0 += 128) {
      int l[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = i0 + k * 32 + lane;
        l[k] = i < ns ? lp[i] : 0;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        int v = l[k];
        if (v < 0) { local_flags |= DSF_FLAG_NEG_LENGTH; v = 0; }
        if (v > kMaxBagLen) { local_flags |= DSF_FLAG_COUNT; v = kMaxBagLen; }
        s += v;
      }
    }
    s = warp_sum(s);
    if (s > 0x7fffffffll) { local_flags |= DSF_FLAG_COUNT; s = 0x7fffffffll; }
    if (lane == 0) {
      st_relaxed_u64(&p.partials[(long long)cta * kMaxF + f], tag | (unsigned long long)s);
    }
  }
  if (ns > 0 && long0) pool_map(nb0, 0, min(U0, (long long)pool_cap(nb0)));

  // ---------------------------------------------------------------- sequence offset
  // First sequence value index of sample sb0: sum of the full lengths before
  // it (this thread's part; the first batch setup adds the parts up).
  long long seq_part = 0;
  if constexpr (C::ATTN) {
#pragma unroll
    for (int k = 0; k < 4; ++k) seq_part += max(seq_pre[k], 0);  // first pass, loaded early
    for (int b0 = 4 * kThreads; b0 < sb0; b0 += 4 * kThreads) {
      int l[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int b = b0 + k * kThreads + tid;
        l[k] = b < sb0 ? p.seq_lengths[b] : 0;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) seq_part += max(l[k], 0);
    }
  }

  // ---------------------------------------------------------------- batch setup
  // Valid-row prefix rp[] and sequence value offsets so[] for samples [bs, be).
  // The first batch takes its lengths from seq_len0 and starts at the sum of
  // the seq_part of all threads; later batches continue from seq_cur.
  auto setup_batch = [&](int bs, int be) {
    const bool first = bs == sb0;
    const int nb = be - bs;
    long long lv = 0, lf = 0;
    if (tid < nb) {
      const int L = first ? seq_len0 : p.seq_lengths[bs + tid];
      if (L < 0) local_flags |= DSF_FLAG_NEG_LENGTH;
      if (L > p.max_len) local_flags |= DSF_FLAG_SEQ_TRUNC;
      lf = max(L, 0);
      lv = min(lf, (long long)p.max_len);
    }
    long long ev, ef, tv, tf, tc;
    block_scan2_sum(lv, lf, first ? seq_part : 0ll, ms->scan64, ms->cred, ev, ef, tv, tf, tc);
    const long long base = first ? tc : ms->seq_cur;
    if (tid < nb) {
      ms->rp[tid] = int(ev);
      const long long so = base + ef;
      ms->so[tid] = so < p.n_seq ? int(so) : int(p.n_seq);
    }
    if (tid == 0) ms->rp[nb] = int(tv);
    __syncthreads();
    // read again only by the next batch's setup, many barriers later
    if (tid == 0) ms->seq_cur = base + tf;
  };

  // The row of an id of table f: the id itself, or, for a table served by the
  // hash table, the pool slot of its raw key (the zero row when unseen,
  // hash::kBadKey -- flagged as out of range below -- for an invalid key).
  auto rid = [&](int f, long long id) -> long long {
    return ((p.hash_mask >> f) & 1u) ? hash::find(p.hkeys, p.hbmask, p.kspace[f], id) : id;
  };
  // Sequence rows of a tile [t0, t0+n): thread tid = 32 + ri, ri < 3n, owns
  // sub-row (r = ri/3, key k = ri%3); warp 0 has none, so that its thread 0
  // can issue MMAs meanwhile. seq_ids finds the row's sample (written once
  // per tile to the ring slot (t0/TM) % 4 by the k = 0 thread) and value index
  // and loads the id; only the id stays in a register until the row copy.
  // kNoRow marks a thread without a row.
  constexpr long long kNoRow = (long long)(~0ull >> 1) * -1 - 1;
  const int ri = tid - 32;
  auto seq_ids = [&](int t0, int n, int nb) -> long long {
    long long id = kNoRow;
    if (ri >= 0 && ri < 3 * n) {
      const int r = ri / 3, k = ri - 3 * r;
      const int rr = t0 + r;
      const int i = upper_index(ms->rp, nb + 1, rr);
      const long long jj = (long long)ms->so[i] + (rr - ms->rp[i]);
      const int j = jj < p.n_seq ? int(jj) : -1;
      if (k == 0) ms->row_samp[(t0 / C::TM) & 3][r] = uint8_t(i);
      if (j >= 0) id = rid(p.seq_table[k], p.seq_values[(long long)k * p.n_seq + j]);
      else local_flags |= DSF_FLAG_COUNT;
    }
    return id;
  };
  // seq_ids of two tiles at once, the two row -> sample searches interleaved
  auto seq_ids2 = [&](int t0a, int na, int t0b, int nbt, int nb, long long& ida, long long& idb) {
    ida = idb = kNoRow;
    if (ri < 0 || ri >= 3 * na) return;
    const int r = ri / 3, k = ri - 3 * r;
    const bool vb = ri < 3 * nbt;
    const int xa = t0a + r, xb = t0b + r;
    int loa = 0, hia = nb, lob = 0, hib = vb ? nb : 0;
    while (loa < hia || lob < hib) {
      if (loa < hia) {
        const int mid = (loa + hia + 1) >> 1;
        if (ms->rp[mid] <= xa) loa = mid; else hia = mid - 1;
      }
      if (lob < hib) {
        const int mid = (lob + hib + 1) >> 1;
        if (ms->rp[mid] <= xb) lob = mid; else hib = mid - 1;
      }
    }
    auto finish = [&](int t0, int xr, int i, long long& id) {
      const long long jj = (long long)ms->so[i] + (xr - ms->rp[i]);
      const int j = jj < p.n_seq ? int(jj) : -1;
      if (k == 0) ms->row_samp[(t0 / C::TM) & 3][r] = uint8_t(i);
      if (j >= 0) id = rid(p.seq_table[k], p.seq_values[(long long)k * p.n_seq + j]);
      else local_flags |= DSF_FLAG_COUNT;
    };
    finish(t0a, xa, loa, ida);
    if (vb) finish(t0b, xb, lob, idb);
  };
  auto s_buf = [&](int buf) -> uint8_t* { return sm + (buf ? C::S1_OFF : C::S_OFF); };
  // The row copy (L1-allocating cp.async) behind a prefetched id; a thread
  // whose row has no value (or an id out of range) zero-fills its piece.
  auto seq_rows = [&](long long id, int n, int buf) {
    if (ri >= 0 && ri < 3 * n) {
      const int r = ri / 3, k = ri - 3 * r;
      const int tb = p.seq_table[k];
      const uint8_t* base = static_cast<const uint8_t*>(p.tables[tb]);
      const bool ok = id >= 0 && id < p.rows[tb];
      if (!ok && id != kNoRow) local_flags |= DSF_FLAG_ID_RANGE;
      uint8_t* dst = s_buf(buf) + r * C::SROWB + k * C::ROWB;
      const uint8_t* src = ok ? base + id * C::ROWB : base;
#pragma unroll
      for (int q = 0; q < C::LPB; ++q) cp_async_16_ca(dst + 16 * q, src + 16 * q, ok ? 16u : 0u);
    }
    cp_async_commit();
  };
  // L2 prefetch of the rows behind a prefetched id (key ri % 3 of row ri / 3).
  auto seq_prefetch = [&](long long id) {
    if (id < 0) return;
    const int tb = p.seq_table[ri % 3];
    if (id >= p.rows[tb]) return;
    const uint8_t* row = static_cast<const uint8_t*>(p.tables[tb]) + id * C::ROWB;
#pragma unroll
    for (int o = 0; o < C::ROWB; o += 128) prefetch_l2(row + o);
  };
  // Exchange of every CTA's per-feature totals: row c of the partials holds
  // CTA c's tagged totals. Thread t reads 16 bytes (features f0 = 2*(t%TPR) and
  // f0+1) of row t/TPR + k*RPP for each of NSLOT slots; TPR = 8 threads per
  // row when F <= 16 (a 128-byte line), else 16. The first pass is issued
  // here and checked after the batch setup, whose work hides its latency.
  const int xsh = F <= 16 ? 3 : 4;
  const int xjp = tid & ((1 << xsh) - 1);
  const int xf0 = 2 * xjp;
  const bool xw0 = xf0 < F, xw1 = xf0 + 1 < F;
  const int xrpp = kThreads >> xsh;
  constexpr int NSLOT = 5;
  unsigned long long xv[NSLOT][2];
  auto exch_issue = [&](int r0) {
#pragma unroll
    for (int k = 0; k < NSLOT; ++k) {
      const int c = r0 + k * xrpp + (tid >> xsh);
      if (c < G && xw0) {
        const ulonglong2 x = ld_relaxed_u64x2(&p.partials[(long long)c * kMaxF + xf0]);
        xv[k][0] = x.x;
        xv[k][1] = x.y;
      } else {
        xv[k][0] = xv[k][1] = tag;
      }
    }
  };
  auto exch_ready = [&]() -> bool {
    bool ready = true;
#pragma unroll
    for (int k = 0; k < NSLOT; ++k)
      ready = ready && (!xw0 || (xv[k][0] & 0xffffffff00000000ull) == tag) &&
              (!xw1 || (xv[k][1] & 0xffffffff00000000ull) == tag);
    return ready;
  };
  exch_issue(0);

  // The first batch's sequence rows: the ids of its first (two) tiles are
  // loaded while pooling waits for its own ids, and the rows of tile 0 are
  // copied into S0 (those of tile 1 prefetched into L2) while pooling waits
  // for its rows.
  bool prefetched = false;
  long long first_id = -1, second_id = -1;
  int first_n = 0, second_n = 0;
  if constexpr (C::ATTN) {
    if (ns > 0) {
      const int be = min(sb0 + kSB, sb1);
      setup_batch(sb0, be);
      const int R0 = ms->rp[be - sb0];
      if (attn_ok && R0 > 0) {
        first_n = min(C::TM, R0);
        if (C::TWO_S && R0 > C::TM) second_n = min(C::TM, R0 - C::TM);
        prefetched = true;
      }
    }
  }
  bool first_ids_todo = prefetched, first_rows_todo = prefetched;
  auto first_ids = [&]() {
    if (!first_ids_todo) return;
    first_ids_todo = false;
    if (second_n > 0) seq_ids2(0, first_n, C::TM, second_n, nb0, first_id, second_id);
    else first_id = seq_ids(0, first_n, nb0);
  };
  auto first_rows = [&]() {
    first_ids();
    if (!first_rows_todo) return;
    first_rows_todo = false;
    seq_rows(first_id, first_n, 0);
    if (C::TWO_S) seq_prefetch(second_id);  // tile 1 lands in S1 after pooling
  };

  // ---------------------------------------------------------------- exchange
  // Wait until every row read carries this launch's tag, then sum the totals
  // (all rows) and the prefix (rows of CTAs before this one) per feature.
  {
    long long tot0 = 0, tot1 = 0, pre0 = 0, pre1 = 0;
    bool ok = true;
    uint64_t t0 = 0;
    for (int r0 = 0; r0 < G; r0 += xrpp * NSLOT) {
      if (r0 > 0) exch_issue(r0);
      while (true) {
        if (__syncthreads_and(exch_ready())) break;
        if (t0 == 0) t0 = globaltimer_ns();
        if (__syncthreads_or(globaltimer_ns() - t0 > kWaitLimitNs)) {
          ok = false;
          break;
        }
        __nanosleep(64);
        exch_issue(r0);
      }
      if (!ok) break;
#pragma unroll
      for (int k = 0; k < NSLOT; ++k) {
        const int c = r0 + k * xrpp + (tid >> xsh);
        if (c >= G) continue;
        const long long x0 = xw0 ? (long long)(xv[k][0] & 0xffffffffull) : 0;
        const long long x1 = xw1 ? (long long)(xv[k][1] & 0xffffffffull) : 0;
        tot0 += x0;
        tot1 += x1;
        if (c < cta) {
          pre0 += x0;
          pre1 += x1;
        }
      }
    }
    // the rows a warp reads share feature pairs: fold lanes l, l + TPR, ...
    for (int off = 1 << xsh; off < 32; off <<= 1) {
      tot0 += __shfl_xor_sync(0xffffffffu, tot0, off);
      tot1 += __shfl_xor_sync(0xffffffffu, tot1, off);
      pre0 += __shfl_xor_sync(0xffffffffu, pre0, off);
      pre1 += __shfl_xor_sync(0xffffffffu, pre1, off);
    }
    if (lane < (1 << xsh)) {
      if (xw0) {
        atomicAdd(reinterpret_cast<unsigned long long*>(&ms->ft[xf0]), (unsigned long long)tot0);
        atomicAdd(reinterpret_cast<unsigned long long*>(&ms->fpre[xf0]), (unsigned long long)pre0);
      }
      if (xw1) {
        atomicAdd(reinterpret_cast<unsigned long long*>(&ms->ft[xf0 + 1]), (unsigned long long)tot1);
        atomicAdd(reinterpret_cast<unsigned long long*>(&ms->fpre[xf0 + 1]), (unsigned long long)pre1);
      }
    }
    if (!ok && tid == 0) ms->abort_ = 1;
    // Every CTA read the epoch before it published its totals, and none reads
    // it again: once CTA 0 has seen all totals it advances the epoch (which
    // tags the next launch's totals). On a timeout it advances it too.
    if (cta == 0 && tid == 0) atomicAdd(p.epoch, 1u);
  }
  // the first tile's row copies go out once the exchange no longer competes
  // with them for the load pipeline
  __syncthreads();
  const bool aborted = ms->abort_ != 0;
  if (aborted) {
    if (tid == 0) local_flags |= DSF_FLAG_TIMEOUT;
  } else {
    if (warp == 0) {
      // feature f's values start after all values of features < f
      const long long t = lane < F ? (long long)ms->ft[lane] : 0;
      const long long incl = warp_incl_scan(t);
      if (lane < F) ms->fcur[lane] = (long long)ms->fpre[lane] + (incl - t);
      const long long total = __shfl_sync(0xffffffffu, incl, 31);
      if (lane == 0 && cta == 0 && total != p.n_values) local_flags |= DSF_FLAG_COUNT;
    }
    __syncthreads();
  }

  // ---------------------------------------------------------------- batches
  uint32_t mma_phase = 0;
  bool bias_ready = false;  // pipelined tiles: bias K-step operands built
  uint32_t gk = 0;  // W1 K-blocks consumed so far (stream mode)
  bool weights_ready = false;
  bool tc_fail = false;

  for (int bs = sb0; !aborted && bs < sb1; bs += kSB) {
    const int be = min(bs + kSB, sb1);
    const int nb = be - bs;
    if (C::ATTN && bs != sb0) setup_batch(bs, be);

    // ------------------------------------------------------------ pooling
    {
      const int nbag = F * nb;
      const unsigned nb_recip = nb_recip_of(nb);
      auto feat_of = [&](int g) -> int { return int((unsigned(g) * nb_recip) >> 20); };
      uint8_t* stage = sm + C::ACT_OFF;
      uint32_t* offs = pool_offs(nb);
      const int cap = pool_cap(nb);
      bool longbag = long0;
      if (bs != sb0) pool_len_load(bs, nb);
      const long long tot = bs == sb0 ? U0 : pool_scan(nb, longbag, false);
      const long long U = longbag ? tot : 0;  // staged windows only for long bags
      if (!longbag) {
        // Direct: one thread per (bag, 16*PPT-byte part), bags in sample-major
        // order, two in flight per thread; ids then rows straight from global
        // memory, summed in value order, stored as one contiguous piece.
        constexpr int PPT = C::LPB < 4 ? C::LPB : 4;
        constexpr int TPB = C::LPB / PPT;
        constexpr int EPT = PPT * C::EPL;
        const int nitems = nbag * TPB;
        const unsigned f_recip = ((1u << 20) + unsigned(F) - 1u) / unsigned(F);
        for (int it0 = 0; it0 < nitems; it0 += 2 * kThreads) {
          long long va[2], ve[2], id[2];
          int fk[2], ik[2], pk[2];
          bool live[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int item = it0 + k * kThreads + tid;
            const int bi = item / TPB;
            pk[k] = item - bi * TPB;
            ik[k] = int((unsigned(bi) * f_recip) >> 20);
            fk[k] = bi - ik[k] * F;
            live[k] = item < nitems && want_feature(fk[k]);
            va[k] = ve[k] = 0;
            id[k] = -1;
            if (live[k]) {
              const int g = fk[k] * nb + ik[k];
              const uint32_t lo = offs[g], hi = offs[g + 1];
              va[k] = ms->fcur[fk[k]] + (long long)(lo - offs[fk[k] * nb]);
              ve[k] = va[k] + (long long)(hi - lo);
              if (va[k] < ve[k]) {
                if (ve[k] <= p.n_values) id[k] = __ldg(p.values + va[k]);
                else { local_flags |= DSF_FLAG_COUNT; ve[k] = va[k]; }
              }
            }
          }
          if constexpr (C::ATTN) first_ids();  // (their latency overlaps ours)
#pragma unroll
          for (int k = 0; k < 2; ++k)
            if (va[k] < ve[k]) id[k] = rid(fk[k], id[k]);
          // first value of both bags: all row loads in flight before the adds
          // (a bag without a usable first value reads row 0 and adds nothing)
          float acc[2][EPT];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const bool has = va[k] < ve[k];
            const bool ok = has && id[k] >= 0 && id[k] < p.rows[fk[k]];
            if (has && !ok) local_flags |= DSF_FLAG_ID_RANGE;
            const uint8_t* src = static_cast<const uint8_t*>(p.tables[fk[k]]) + (ok ? id[k] : 0) * C::ROWB +
                                 pk[k] * PPT * 16;
#pragma unroll
            for (int q = 0; q < PPT; ++q) {
              float x[C::EPL];
              widen16v<C::BF16>(ldg16(src + 16 * q), x);
#pragma unroll
              for (int e = 0; e < C::EPL; ++e) acc[k][q * C::EPL + e] = 0.f + (ok ? x[e] : 0.f);
            }
          }
          // the rest of each bag, in value order
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            for (long long u = va[k] + 1; u < ve[k]; ++u) {
              const long long v = rid(fk[k], __ldg(p.values + u));
              if (v < 0 || v >= p.rows[fk[k]]) { local_flags |= DSF_FLAG_ID_RANGE; continue; }
              const uint8_t* src = static_cast<const uint8_t*>(p.tables[fk[k]]) + v * C::ROWB + pk[k] * PPT * 16;
#pragma unroll
              for (int q = 0; q < PPT; ++q) {
                float x[C::EPL];
                widen16v<C::BF16>(ldg16(src + 16 * q), x);
#pragma unroll
                for (int e = 0; e < C::EPL; ++e) acc[k][q * C::EPL + e] += x[e];
              }
            }
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            if (!live[k]) continue;
            const long long b = bs + ik[k];
            if ((p.mean_mask >> fk[k]) & 1u) {
              // mean pooling: the fp32 sum over the bag's length (empty stays 0)
              const int g = fk[k] * nb + ik[k];
              const uint32_t L = offs[g + 1] - offs[g];
              if (L > 0) {
#pragma unroll
                for (int q = 0; q < EPT; ++q) acc[k][q] = acc[k][q] / float(L);
              }
            }
            auto put = [&](float* o) {
#pragma unroll
              for (int q = 0; q < EPT; q += 4)
                *reinterpret_cast<float4*>(o + q) = make_float4(acc[k][q], acc[k][q + 1], acc[k][q + 2], acc[k][q + 3]);
            };
            if (pool_all) {
              put(p.pooled + b * F * D + fk[k] * D + pk[k] * EPT);
            } else {
              for (int j = 0; j < 3; ++j)
                if (p.q_feat[j] == fk[k]) put(p.qbuf + b * Q + j * D + pk[k] * EPT);
            }
            if constexpr (C::TWO_S) {
              // the batch's query slices for the attention tiles
              for (int j = 0; j < 3; ++j)
                if (p.q_feat[j] == fk[k])
                  put(reinterpret_cast<float*>(sm + C::ACT_OFF) + ik[k] * C::QROW + j * D + pk[k] * EPT);
            }
          }
        }
        // tile 0's rows into S0 (its ids have landed meanwhile)
        if constexpr (C::ATTN) first_rows();
      }
      if constexpr (C::ATTN) first_rows();  // (staged pooling: before its windows)
      int widx = 0;
      for (long long w0 = 0; w0 < U; w0 += cap, ++widx) {
        const long long w1 = min(U, w0 + (long long)cap);
        // value -> (feature, index) map in the staging slots (the first window
        // of the first batch was mapped before the exchange)
        if (!(bs == sb0 && widx == 0)) {
          pool_map(nb, w0, w1);
          __syncthreads();
        }
        // ids first (all loads in flight), then the row copies
        long long idv[C::VPT];
        int fv[C::VPT];
        bool inw[C::VPT];
#pragma unroll
        for (int k = 0; k < C::VPT; ++k) {
          const long long u = w0 + tid + (long long)k * kThreads;
          inw[k] = false;
          idv[k] = -1;
          fv[k] = 0;
          if (u < w1) {
            const int2 fl = *reinterpret_cast<const int2*>(stage + (u - w0) * C::ROWB);
            const int f = fl.x;
            fv[k] = f;
            if (want_feature(f)) {
              inw[k] = true;
              const long long gv = ms->fcur[f] + fl.y;
              if (gv < p.n_values) idv[k] = p.values[gv];
              else local_flags |= DSF_FLAG_COUNT;
            }
          }
        }
#pragma unroll
        for (int k = 0; k < C::VPT; ++k) {
          if (!inw[k]) continue;
          const long long u = w0 + tid + (long long)k * kThreads;
          const int f = fv[k];
          const uint8_t* tbase = static_cast<const uint8_t*>(p.tables[f]);
          const long long id = rid(f, idv[k]);
          const bool ok = id >= 0 && id < p.rows[f];
          if (!ok) local_flags |= DSF_FLAG_ID_RANGE;
          uint8_t* dst = stage + (u - w0) * C::ROWB;
          const uint8_t* src = ok ? tbase + id * C::ROWB : tbase;
#pragma unroll
          for (int q = 0; q < C::LPB; ++q) cp_async_16_ca(dst + 16 * q, src + 16 * q, ok ? 16u : 0u);
        }
        cp_async_commit();
        cp_async_wait_all();
        __syncthreads();
        // sum the bags that intersect [w0, w1), in value order
        const int ga = upper_index(offs, nbag + 1, w0);
        const int gb = upper_index(offs, nbag + 1, w1 - 1);
        float* cin = ms->pcarry[widx & 1];
        float* cout = ms->pcarry[(widx + 1) & 1];
        const int grp = tid / C::LPB, sub = tid - grp * C::LPB;
        constexpr int NGRP = kThreads / C::LPB;
        for (int g = ga + grp; g <= gb; g += NGRP) {
          const long long a = offs[g], e = offs[g + 1];
          if (a == e) continue;
          const int f = feat_of(g);
          if (!want_feature(f)) continue;
          float acc[C::EPL];
          if (a < w0) {
#pragma unroll
            for (int q = 0; q < C::EPL; ++q) acc[q] = cin[sub * C::EPL + q];
          } else {
#pragma unroll
            for (int q = 0; q < C::EPL; ++q) acc[q] = 0.f;
          }
          const long long lo = a < w0 ? w0 : a, hi = e < w1 ? e : w1;
          for (long long u = lo; u < hi; ++u) {
            float v[C::EPL];
            widen16<C::BF16>(stage + (u - w0) * C::ROWB + sub * 16, v);
#pragma unroll
            for (int q = 0; q < C::EPL; ++q) acc[q] += v[q];
          }
          if (e <= w1) {
            if ((p.mean_mask >> f) & 1u) {
              // mean pooling: the fp32 sum over the bag's length (e > a here)
#pragma unroll
              for (int q = 0; q < C::EPL; ++q) acc[q] = acc[q] / float(e - a);
            }
            const int i = g - f * nb;
            const long long b = bs + i;
            if (pool_all) {
              float* o = p.pooled + b * F * D + f * D + sub * C::EPL;
#pragma unroll
              for (int q = 0; q < C::EPL; q += 4)
                *reinterpret_cast<float4*>(o + q) = make_float4(acc[q], acc[q + 1], acc[q + 2], acc[q + 3]);
            } else {
#pragma unroll
              for (int k = 0; k < 3; ++k) {
                if (p.q_feat[k] != f) continue;
                float* o = p.qbuf + b * Q + k * D + sub * C::EPL;
#pragma unroll
                for (int q = 0; q < C::EPL; q += 4)
                  *reinterpret_cast<float4*>(o + q) = make_float4(acc[q], acc[q + 1], acc[q + 2], acc[q + 3]);
              }
            }
          } else {
#pragma unroll
            for (int q = 0; q < C::EPL; ++q) cout[sub * C::EPL + q] = acc[q];
          }
        }
        __syncthreads();
      }
      // empty bags
      for (int g = tid; longbag && g < nbag; g += kThreads) {
        if (offs[g] != offs[g + 1]) continue;
        const int f = g / nb, i = g - f * nb;
        if (!want_feature(f)) continue;
        const long long b = bs + i;
        if (pool_all) {
          float* o = p.pooled + b * F * D + f * D;
          for (int q = 0; q < D; q += 4) *reinterpret_cast<float4*>(o + q) = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
          for (int k = 0; k < 3; ++k) {
            if (p.q_feat[k] != f) continue;
            float* o = p.qbuf + b * Q + k * D;
            for (int q = 0; q < D; q += 4) *reinterpret_cast<float4*>(o + q) = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      }
      __syncthreads();
      if constexpr (C::TWO_S) {
        if (longbag) {
          // staged pooling wrote the query slices to global memory only
          constexpr int P4 = D / 4;
          for (int it = tid; it < nb * 3 * P4; it += kThreads) {
            const int i = it / (3 * P4), rem = it - i * 3 * P4, j = rem / P4, q = rem - j * P4;
            const float* src = pool_all ? p.pooled + (long long)(bs + i) * F * D + p.q_feat[j] * D
                                        : p.qbuf + (long long)(bs + i) * Q + j * D;
            cp_async_16_ca(reinterpret_cast<float*>(sm + C::ACT_OFF) + i * C::QROW + j * D + 4 * q, src + 4 * q, 16u);
          }
          cp_async_commit();
          cp_async_wait_all();
        }
      }
      if (tid < F) ms->fcur[tid] += (long long)offs[(tid + 1) * nb] - (long long)offs[tid * nb];
      __syncthreads();
    }

    if constexpr (C::ATTN) {
      if (!attn_ok || tc_fail) continue;
      // samples without a valid position get zeros
      for (int i = tid; i < nb; i += kThreads) {
        if (ms->rp[i] != ms->rp[i + 1]) continue;
        float* o = p.din + (long long)(bs + i) * Q;
        for (int d = 0; d < Q; d += 4) *reinterpret_cast<float4*>(o + d) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      const int R = ms->rp[nb];
      const int T = (R + C::TM - 1) / C::TM;  // tiles of this batch
      if (!C::TWO_S && T > 0 && !(prefetched && bs == sb0))
        seq_rows(seq_ids(0, min(C::TM, R), nb), min(C::TM, R), 0);
      if (T == 0) continue;

      // masked softmax + weighted sum of tile [t0, t0+n) held in S buffer `buf`.
      // (1) Per sample segment of the tile, a group of 8 lanes: the running max
      // m over its valid rows (merged with the state carried from the previous
      // tile), z[r] <- exp(z[r] - m) and l = sum of those. (2) One thread per
      // (segment, 4 consecutive d): sum_r exp(z_r - m) s[r][d] over the
      // segment's rows with two interleaved partial sums. A segment that continues into the next
      // tile hands (m, l, acc) on. With skip0, warp 0 takes no part (its thread
      // 0 is issuing MMAs).
      auto softmax_tile = [&](int t0, int n, int tix, int buf, bool skip0) {
        const uint8_t* S = s_buf(buf);
        const int slot = tix & 3;
        const int ia = ms->row_samp[slot][0], ib = ms->row_samp[slot][n - 1];
        const int nseg = ib - ia + 1;
        const float* cin = ms->carry[tix & 1];
        float* cout = ms->carry[(tix + 1) & 1];
        float* z = ms->z;
        float* seg_sc = ms->red[0];   // scale of the carried-in state
        float* seg_inv = ms->red[1];  // 1 / l, or 0 when the segment carries out
        float* seg_m = ms->red[2];
        float* seg_l = ms->red[3];
        const int t_lo = skip0 ? 32 : 0;
        if (p.logits) {
          for (int r = tid; r < n; r += kThreads) {
            const int i = ms->row_samp[slot][r];
            const long long j = (long long)ms->so[i] + (t0 + r - ms->rp[i]);
            if (j < p.n_seq) p.logits[j] = z[r];
          }
          __syncthreads();
        }
        if (tid >= t_lo) {
          const int gl = lane & 7;
          const unsigned gmask = 0xffu << (lane & 24);
          const int ngrp = (kThreads - t_lo) >> 3;
          for (int g = (tid - t_lo) >> 3; g < nseg; g += ngrp) {
            const int si = ia + g;
            const int ra = ms->rp[si], re = ms->rp[si + 1];
            const int r0 = max(ra, t0) - t0, r1 = min(re, t0 + n) - t0;
            if (r1 <= r0) continue;
            const bool has_in = ra < t0, has_out = re > t0 + n;
            float m = -INFINITY;
            for (int r = r0 + gl; r < r1; r += 8) m = fmaxf(m, z[r]);
            m = fmaxf(m, __shfl_xor_sync(gmask, m, 4));
            m = fmaxf(m, __shfl_xor_sync(gmask, m, 2));
            m = fmaxf(m, __shfl_xor_sync(gmask, m, 1));
            if (has_in) m = fmaxf(m, cin[0]);
            float l = 0.f;
            for (int r = r0 + gl; r < r1; r += 8) {
              const float e = expf(z[r] - m);
              z[r] = e;
              l += e;
            }
            l += __shfl_xor_sync(gmask, l, 4);
            l += __shfl_xor_sync(gmask, l, 2);
            l += __shfl_xor_sync(gmask, l, 1);
            if (gl == 0) {
              const float sc = has_in ? expf(cin[0] - m) : 0.f;
              if (has_in) l += cin[1] * sc;
              seg_sc[g] = sc;
              seg_inv[g] = has_out ? 0.f : 1.f / l;
              seg_m[g] = m;
              seg_l[g] = l;
            }
          }
        }
        __syncthreads();
        const int stride = kThreads - t_lo;
        constexpr int Q4 = Q / 4;
        for (int item = tid - t_lo; item >= 0 && item < nseg * Q4; item += stride) {
          const int g = item / Q4, d = (item - g * Q4) * 4;
          const int si = ia + g;
          const int ra = ms->rp[si], re = ms->rp[si + 1];
          const int r0 = max(ra, t0) - t0, r1 = min(re, t0 + n) - t0;
          if (r1 <= r0) continue;
          const bool has_in = ra < t0, has_out = re > t0 + n;
          // two interleaved partial sums (even / odd rows of the segment)
          float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
          int r = r0;
          for (; r + 2 <= r1; r += 2) {
            const float e0 = z[r], e1 = z[r + 1];
            const float4 s0 = s_quad<C::BF16>(S, C::SROWB, r, d), s1 = s_quad<C::BF16>(S, C::SROWB, r + 1, d);
            a.x = fmaf(e0, s0.x, a.x); a.y = fmaf(e0, s0.y, a.y); a.z = fmaf(e0, s0.z, a.z); a.w = fmaf(e0, s0.w, a.w);
            b.x = fmaf(e1, s1.x, b.x); b.y = fmaf(e1, s1.y, b.y); b.z = fmaf(e1, s1.z, b.z); b.w = fmaf(e1, s1.w, b.w);
          }
          if (r < r1) {
            const float e0 = z[r];
            const float4 s0 = s_quad<C::BF16>(S, C::SROWB, r, d);
            a.x = fmaf(e0, s0.x, a.x); a.y = fmaf(e0, s0.y, a.y); a.z = fmaf(e0, s0.z, a.z); a.w = fmaf(e0, s0.w, a.w);
          }
          float4 acc = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
          if (has_in) {
            const float sc = seg_sc[g];
            const float4 c = *reinterpret_cast<const float4*>(cin + 4 + d);
            acc = make_float4(fmaf(c.x, sc, acc.x), fmaf(c.y, sc, acc.y), fmaf(c.z, sc, acc.z), fmaf(c.w, sc, acc.w));
          }
          if (has_out) {
            *reinterpret_cast<float4*>(cout + 4 + d) = acc;
            if (d == 0) {
              cout[0] = seg_m[g];
              cout[1] = seg_l[g];
            }
          } else {
            const float inv = seg_inv[g];
            *reinterpret_cast<float4*>(p.din + (long long)(bs + si) * Q + d) =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
          }
        }
        __syncthreads();
      };

      if constexpr (C::STREAM) {
        // ---------------------------------------------------------- streamed W1 (D = 64)
        // Per tile: 12 K-blocks of layer 1. x K-block kb (part kb/3 of
        // cat[q, s, q-s, q*s], dims (kb%3)*64..+64) is built in x-ring slot kb%2;
        // W1 K-block kb arrives in W1-ring slot gk%3 by bulk copy (gk counts
        // blocks over the whole launch). Thread 0 issues each block's 4 MMAs,
        // commits them to the slot's done barrier and refills the slot of the
        // previous block once its MMAs are done.
        const uint32_t tbase = ms->tmem_base;
        const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
        const bool pa = p.pooled != nullptr;
        const float* qsrc = pa ? p.pooled : p.qbuf;
        const long long qstride = pa ? (long long)F * D : Q;
        constexpr int NKB = C::K1 / 64;
        auto load_w1 = [&](uint32_t g) {  // thread 0
          const int slot = int(g % 3u), blk = int(g % uint32_t(NKB));
          mbar_arrive_expect_tx(&ms->mbar_full[slot], C::W1KB);
          for (int off = 0; off < C::W1KB; off += 16384)
            bulk_g2s(sm + C::W1_OFF + slot * C::W1KB + off, p.wpack + (size_t)blk * C::W1KB + off, 16384,
                     &ms->mbar_full[slot]);
        };
        for (int t0 = 0, tix = 0; t0 < R && !tc_fail; t0 += C::TM, ++tix) {
          const int n = min(C::TM, R - t0);
          cp_async_wait_all();
          __syncthreads();
          const int t1 = t0 + C::TM;
          const bool has_next = t1 < R;
          long long nxt = -1;
          if (has_next) nxt = seq_ids(t1, min(C::TM, R - t1), nb);
          const uint8_t* S = s_buf(0);
          if (tid == 0) {
            load_w1(gk);
            load_w1(gk + 1);
          }
          for (int kb = 0; kb < NKB; ++kb, ++gk) {
            uint8_t* X = sm + C::XR_OFF + (kb & 1) * C::XKB;
            const int part = kb / 3, k = kb % 3;
            for (int item = tid; item < n * 8; item += kThreads) {
              const int r = item >> 3, c = item & 7;
              uint4 out = make_uint4(0u, 0u, 0u, 0u);
              {
                const long long b = bs + ms->row_samp[tix & 3][r];
                float qv[8], sv[8];
                if (part != 1) {
                  const float* qp = qsrc + b * qstride + (pa ? p.q_feat[k] * D : k * D) + c * 8;
                  const float4 a = *reinterpret_cast<const float4*>(qp);
                  const float4 a2 = *reinterpret_cast<const float4*>(qp + 4);
                  qv[0] = a.x; qv[1] = a.y; qv[2] = a.z; qv[3] = a.w;
                  qv[4] = a2.x; qv[5] = a2.y; qv[6] = a2.z; qv[7] = a2.w;
                }
                if (part != 0) widen16<true>(S + r * C::SROWB + (k * 64 + c * 8) * 2, sv);
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  float x0, x1;
                  if (part == 0) { x0 = qv[2 * e]; x1 = qv[2 * e + 1]; }
                  else if (part == 1) { x0 = sv[2 * e]; x1 = sv[2 * e + 1]; }
                  else if (part == 2) { x0 = qv[2 * e] - sv[2 * e]; x1 = qv[2 * e + 1] - sv[2 * e + 1]; }
                  else { x0 = qv[2 * e] * sv[2 * e]; x1 = qv[2 * e + 1] * sv[2 * e + 1]; }
                  w[e] = pack_bf16x2(x0, x1);
                }
                out = make_uint4(w[0], w[1], w[2], w[3]);
              }
              *reinterpret_cast<uint4*>(X + sw128_offset(uint32_t(r), uint32_t(c * 8), C::TM)) = out;
            }
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
              const int slot = int(gk % 3u);
              bool ok = mbar_wait(&ms->mbar_full[slot], (gk / 3u) & 1u);
              if (ok) {
                tc_fence_after();
                constexpr uint32_t IDESC1 = idesc_bf16_f32(128, kN1);
                const uint32_t xa = smem_u32(X), wa = smem_u32(sm + C::W1_OFF + slot * C::W1KB);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  tc_mma_f16(tbase + C::TM_ACC1, sw128_kmajor_desc(xa + kk * 32), sw128_kmajor_desc(wa + kk * 32),
                             IDESC1, (kb > 0 || kk > 0) ? 1u : 0u);
                tc_commit(&ms->mbar_done[slot]);
                if (kb >= 1) ok = mbar_wait(&ms->mbar_done[(gk - 1u) % 3u], ((gk - 1u) / 3u) & 1u);
                if (ok && kb + 2 < NKB) load_w1(gk + 2u);
              }
              ms->abort_ = ok ? 0 : 3;
            }
            __syncthreads();
            if (ms->abort_ != 0) { tc_fail = true; break; }
          }
          if (tc_fail) break;
          // all of layer 1 done (the last block's commit covers every earlier MMA)
          if (tid == 0) {
            bool ok = mbar_wait(&ms->mbar_done[(gk - 1u) % 3u], ((gk - 1u) / 3u) & 1u);
            if (ok && !weights_ready) ok = mbar_wait(&ms->mbar_w, 0);
            weights_ready = weights_ready || ok;
            ms->abort_ = ok ? 0 : 3;
          }
          __syncthreads();
          if (ms->abort_ != 0) { tc_fail = true; break; }
          tc_fence_after();
          // epilogue 1: h1 packed in place over the first half of each group's columns
          if ((warp & 3) * 32 < n) {
            const int cg = warp >> 2;
            const uint32_t ta = tbase + lane_base + C::TM_ACC1 + uint32_t(cg * 64);
#pragma unroll 1
            for (int qq = 0; qq < 4; ++qq) {
              float v[16];
              tmem_ld16(ta + qq * 16, v);
              tmem_ld_wait();
              uint32_t h[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int col = cg * 64 + qq * 16 + 2 * e;
                h[e] = pack_bf16x2(fmaxf(v[2 * e] + ms->b1[col], 0.f), fmaxf(v[2 * e + 1] + ms->b1[col + 1], 0.f));
              }
              tmem_st8(ta + qq * 8, h);
            }
            tmem_st_wait();
          }
          tc_fence_before();
          __syncthreads();
          if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t IDESC2 = idesc_bf16_f32(128, kN2);
            const uint32_t wa = smem_u32(sm + C::W2_OFF);
#pragma unroll
            for (int kk = 0; kk < kN1 / 16; ++kk) {
              const uint32_t kb2 = kk >> 2, ko = (kk & 3) * 32;
              tc_mma_f16_ts(tbase + C::TM_ACC2, tbase + C::TM_ACC1 + kb2 * 64 + uint32_t((kk & 3) * 8),
                            sw128_kmajor_desc(wa + kb2 * kN2 * 128 + ko), IDESC2, kk > 0);
            }
            tc_commit(&ms->mbar_mma);
            ms->abort_ = mbar_wait(&ms->mbar_mma, mma_phase) ? 0 : 3;
          }
          mma_phase ^= 1u;
          __syncthreads();
          if (ms->abort_ != 0) { tc_fail = true; break; }
          tc_fence_after();
          if ((warp & 3) * 32 < n) {
            const int cg = warp >> 2;
            float v[16];
            tmem_ld16(tbase + lane_base + C::TM_ACC2 + uint32_t(cg * 16), v);
            tmem_ld_wait();
            float part = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int col = cg * 16 + e;
              part += fmaxf(v[e] + ms->b2[col], 0.f) * ms->w3[col];
            }
            ms->red[cg][(warp & 3) * 32 + lane] = part;
          }
          tc_fence_before();
          __syncthreads();
          if (tid < C::TM) ms->z[tid] = ((ms->red[0][tid] + ms->red[1][tid]) + (ms->red[2][tid] + ms->red[3][tid])) + b3;
          __syncthreads();
          softmax_tile(t0, n, tix, 0, false);
          if (has_next) seq_rows(nxt, min(C::TM, R - t1), 0);
        }
      } else if constexpr (C::MODE == 0) {
        // ---------------------------------------------------------- pipelined tiles
        // Per tile k: wait layer 1 (k); epilogue 1 (h1 -> TMEM); issue layer 2 (k);
        // build x (k+1) while it runs; wait layer 2; epilogue 2 (z); issue layer 1
        // (k+1); softmax (k) while it runs; copy the rows of tile k+2 into the
        // freed buffer. Rows run two tiles ahead (in L2 three), their ids three.
        // The query slices of every sample of the batch sit in QS (pooling put
        // them there).
        const uint32_t tbase = ms->tmem_base;
        const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
        const float* QS = reinterpret_cast<const float*>(sm + C::ACT_OFF);  // [kSB][QROW]
        // x tile -> tensor memory: warp w builds part w/4 of cat[q, s, q-s, q*s]
        // for rows 32*(w%4) .. +31, 8 dims (4 packed columns) at a time
        auto build_x = [&](int n, int buf, int slot) {
          if ((warp & 3) * 32 >= n) return;  // rows past the tile end are never read back
          const uint8_t* S = s_buf(buf);
          const int part = warp >> 2;
          const int r = (warp & 3) * 32 + lane;
          const bool live = r < n;
          const float* qrow = QS + (live ? ms->row_samp[slot][r] : 0) * C::QROW;
          const uint8_t* srow = S + r * C::SROWB;
          const uint32_t xa = tbase + lane_base + C::TM_X + uint32_t(part * (Q / 2));
#pragma unroll 2
          for (int c = 0; c < Q / 8; ++c) {
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            if (live) {
              float qv[8], sv[8];
              if (part != 1) {
                const float4 a = *reinterpret_cast<const float4*>(qrow + c * 8);
                const float4 b2 = *reinterpret_cast<const float4*>(qrow + c * 8 + 4);
                qv[0] = a.x; qv[1] = a.y; qv[2] = a.z; qv[3] = a.w;
                qv[4] = b2.x; qv[5] = b2.y; qv[6] = b2.z; qv[7] = b2.w;
              }
              if (part != 0) {
#pragma unroll
                for (int i = 0; i < 8 / C::EPL; ++i)
                  widen16<C::BF16>(srow + (c * 8 + i * C::EPL) * C::ES, sv + i * C::EPL);
              }
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float x0, x1;
                if (part == 0) { x0 = qv[2 * e]; x1 = qv[2 * e + 1]; }
                else if (part == 1) { x0 = sv[2 * e]; x1 = sv[2 * e + 1]; }
                else if (part == 2) { x0 = qv[2 * e] - sv[2 * e]; x1 = qv[2 * e + 1] - sv[2 * e + 1]; }
                else { x0 = qv[2 * e] * sv[2 * e]; x1 = qv[2 * e + 1] * sv[2 * e + 1]; }
                w[e] = pack_bf16x2(x0, x1);
              }
            }
            tmem_st4(xa + uint32_t(c * 4), w);
          }
          tmem_st_wait();
        };
        auto issue_l1 = [&]() {  // thread 0
          tc_fence_after();
          constexpr uint32_t IDESC1 = idesc_bf16_f32(128, kN1);
          const uint32_t wa = smem_u32(sm + C::W1_OFF);
#pragma unroll
          for (int kk = 0; kk < C::K1 / 16; ++kk) {
            const uint32_t kb = kk >> 2, ko = (kk & 3) * 32;
            tc_mma_f16_ts(tbase + C::TM_ACC1, tbase + C::TM_X + uint32_t(kk * 8),
                          sw128_kmajor_desc(wa + kb * kN1 * 128 + ko), IDESC1, kk > 0);
          }
          // + b1: one more K-step, (1, 1, 0 ...) against (b1_hi, b1_lo, 0 ...)
          tc_mma_f16_ts(tbase + C::TM_ACC1, tbase + C::TM_ONE, sw32_kmajor_desc(smem_u32(sm + C::BIAS_OFF)),
                        IDESC1, 1u);
          tc_commit(&ms->mbar_mma);
        };
        // h1 of hidden units [64g, 64g+64) sits packed in accumulator columns
        // [64g, 64g+32): K-step kk of layer 2 reads columns 64(kk/4) + 8(kk%4)
        auto issue_l2 = [&]() {  // thread 0
          tc_fence_after();
          constexpr uint32_t IDESC2 = idesc_bf16_f32(128, kN2);
          const uint32_t wa = smem_u32(sm + C::W2_OFF);
#pragma unroll
          for (int kk = 0; kk < kN1 / 16; ++kk) {
            const uint32_t kb = kk >> 2, ko = (kk & 3) * 32;
            tc_mma_f16_ts(tbase + C::TM_ACC2, tbase + C::TM_ACC1 + kb * 64 + uint32_t((kk & 3) * 8),
                          sw128_kmajor_desc(wa + kb * kN2 * 128 + ko), IDESC2, kk > 0);
          }
          // + b2, as for layer 1
          tc_mma_f16_ts(tbase + C::TM_ACC2, tbase + C::TM_ONE,
                        sw32_kmajor_desc(smem_u32(sm + C::BIAS_OFF + C::BIAS1B)), IDESC2, 1u);
          tc_commit(&ms->mbar_mma);
        };
        // one thread waits for the MMAs, the block learns the outcome together
        auto wait_mma = [&]() -> bool {
          if (tid == 0) ms->abort_ = mbar_wait(&ms->mbar_mma, mma_phase) ? 0 : 3;
          mma_phase ^= 1u;
          __syncthreads();
          if (ms->abort_ != 0) return false;
          tc_fence_after();
          return true;
        };

        // prologue: rows of tile 0 are in S0 (or on their way); x (0), then
        // layer 1 (0) from thread 0 while warps 1.. send out the rows of tile 1
        // (already in L2 for the first batch) and the ids of tile 2
        auto tile_n = [&](int kt) { return min(C::TM, R - kt * C::TM); };
        long long id1 = -1, nxt = -1;
        if (prefetched && bs == sb0) {
          id1 = second_id;
        } else {
          seq_rows(seq_ids(0, tile_n(0), nb), tile_n(0), 0);
          if (T > 1) id1 = seq_ids(C::TM, tile_n(1), nb);
        }
        cp_async_wait_all();
        __syncthreads();
        if (!bias_ready) {
          // The bias K-step operands, once per launch (the biases are in smem by
          // now): row n of B holds (b_hi, b_lo, 0 ...) in both 16-byte halves,
          // b_hi = bf16(b), b_lo = bf16(b - b_hi), so that either half read
          // against A's (1, 1, 0 ...) adds b_hi + b_lo (within 2^-17 |b| of b).
          bias_ready = true;
          for (int r = tid; r < kN1 + kN2; r += kThreads) {
            const float b = r < kN1 ? ms->b1[r] : ms->b2[r - kN1];
            const float hi = __bfloat162float(__float2bfloat16_rn(b));
            const uint4 row = make_uint4(pack_bf16x2(hi, b - hi), 0u, 0u, 0u);
            uint4* dst = reinterpret_cast<uint4*>(sm + C::BIAS_OFF + r * 32);
            dst[0] = row;
            dst[1] = row;
          }
          fence_proxy_async_smem();
          if (warp < 4) {
            uint32_t one[8] = {pack_bf16x2(1.f, 1.f), 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            tmem_st8(tbase + lane_base + C::TM_ONE, one);
            tmem_st_wait();
          }
        }
        build_x(min(C::TM, R), 0, 0);
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
          bool ok = true;
          if (!weights_ready) ok = mbar_wait(&ms->mbar_w, 0);
          weights_ready = weights_ready || ok;
          if (ok) issue_l1();
          else ms->abort_ = 2;
        }
        if (T > 1) seq_rows(id1, tile_n(1), 1);
        if (T > 2) nxt = seq_ids(2 * C::TM, tile_n(2), nb);
        __syncthreads();
        if (ms->abort_ != 0) tc_fail = true;

        for (int k = 0; k < T && !tc_fail; ++k) {
          const int buf = k & 1;
          const int t0 = k * C::TM, n = min(C::TM, R - t0);
          // ---- layer 1 (k) done: epilogue 1, h1 packed back into TMEM
          if (!wait_mma()) { tc_fail = true; break; }
          if ((warp & 3) * 32 < n) {
            const int cg = warp >> 2;
            const uint32_t ta = tbase + lane_base + C::TM_ACC1 + uint32_t(cg * 64);
#pragma unroll 1
            for (int qp = 0; qp < 2; ++qp) {
              float v[32];
              tmem_ld16(ta + qp * 32, v);
              tmem_ld16(ta + qp * 32 + 16, v + 16);
              tmem_ld_wait();
              // (b1 is in the accumulator already: ReLU and round to bf16)
              uint32_t h[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) h[e] = pack_bf16x2_relu(v[2 * e], v[2 * e + 1]);
              // columns [64cg + 16qp, +16) were read by this warp already
              tmem_st16(ta + qp * 16, h);
            }
            tmem_st_wait();
          }
          // rows of tile k+2 into L2 now: their copy into S (after the softmax
          // of tile k frees the buffer) then hits L2
          if (k + 2 < T) seq_prefetch(nxt);
          // (the rows of tile k+1 have landed too)
          cp_async_wait_all();
          tc_fence_before();
          __syncthreads();
          if (tid == 0) issue_l2();
          // ---- x of tile k+1 while layer 2 (k) runs
          if (k + 1 < T) {
            build_x(min(C::TM, R - t0 - C::TM), buf ^ 1, (k + 1) & 3);
            tc_fence_before();
          }
          // ---- layer 2 (k) done: epilogue 2, z = w3 . ReLU(acc) + b3 (b2 is in acc)
          if (!wait_mma()) { tc_fail = true; break; }
          if ((warp & 3) * 32 < n) {
            const int cg = warp >> 2;
            float v[16];
            tmem_ld16(tbase + lane_base + C::TM_ACC2 + uint32_t(cg * 16), v);
            tmem_ld_wait();
            float part = 0.f;
#pragma unroll
            for (int e = 0; e < 16; e += 4) {
              const float4 ww = *reinterpret_cast<const float4*>(ms->w3 + cg * 16 + e);
              part += fmaxf(v[e], 0.f) * ww.x;
              part += fmaxf(v[e + 1], 0.f) * ww.y;
              part += fmaxf(v[e + 2], 0.f) * ww.z;
              part += fmaxf(v[e + 3], 0.f) * ww.w;
            }
            ms->red[cg][(warp & 3) * 32 + lane] = part;
          }
          tc_fence_before();
          __syncthreads();
          if (tid < C::TM) ms->z[tid] = ((ms->red[0][tid] + ms->red[1][tid]) + (ms->red[2][tid] + ms->red[3][tid])) + b3;
          __syncthreads();
          // ---- layer 1 (k+1) runs during the softmax of tile k (warp 0 issues it)
          if (tid == 0 && k + 1 < T) issue_l1();
          softmax_tile(t0, n, k, buf, k + 1 < T);
          // ---- rows of tile k+2 into the freed buffer
          if (k + 2 < T) {
            seq_rows(nxt, tile_n(k + 2), buf);
            if (k + 3 < T) nxt = seq_ids(t0 + 3 * C::TM, tile_n(k + 3), nb);
          }
        }
      } else {
        // ---------------------------------------------------------- sequential tiles (fp32)
        for (int t0 = 0, tix = 0; t0 < R; t0 += C::TM, ++tix) {
          const int n = min(C::TM, R - t0);
          cp_async_wait_all();
          __syncthreads();
          const int t1 = t0 + C::TM;
          const bool has_next = t1 < R;
          long long nxt = -1;
          if (has_next) nxt = seq_ids(t1, min(C::TM, R - t1), nb);
          const uint8_t* S = s_buf(0);
          const float* qsrc = pool_all ? p.pooled : p.qbuf;
          const long long qstride = pool_all ? (long long)F * D : Q;
          {
            // ---------------------------------------------- fp32 check mode
            float* QT = reinterpret_cast<float*>(sm + C::QT_OFF);
            float* H1 = reinterpret_cast<float*>(sm + C::ACT_OFF);
            constexpr int Q4 = Q / 4;
            for (int item = tid; item < C::TM * Q4; item += kThreads) {
              const int r = item / Q4, o = item - r * Q4;
              float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
              if (r < n) {
                const long long b = bs + ms->row_samp[tix & 3][r];
                const int d0 = o * 4, k = d0 / D, dd = d0 - k * D;
                v = ldcg4(qsrc + b * qstride + (pool_all ? p.q_feat[k] * D : k * D) + dd);
              }
              *reinterpret_cast<float4*>(QT + r * Q + o * 4) = v;
            }
            __syncthreads();
            {
              // layer 1: thread = 4 rows x 8 units
              const int rg = warp, ug = lane;
              float acc[4][8];
  #pragma unroll
              for (int a = 0; a < 4; ++a)
  #pragma unroll
                for (int u = 0; u < 8; ++u) acc[a][u] = 0.f;
              auto run_part = [&](auto part_tag) {
                constexpr int PART = decltype(part_tag)::value;
                for (int d = 0; d < Q; ++d) {
                  const float* wp = p.w1t + (long long)(PART * Q + d) * kN1 + ug * 8;
                  const float4 wa = __ldg(reinterpret_cast<const float4*>(wp));
                  const float4 wb = __ldg(reinterpret_cast<const float4*>(wp + 4));
                  const float w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
  #pragma unroll
                  for (int a = 0; a < 4; ++a) {
                    const int r = rg * 4 + a;
                    const float qv = QT[r * Q + d];
                    const float sv = s_elem<C::BF16>(S, C::SROWB, r, d);
                    float x;
                    if constexpr (PART == 0) x = qv;
                    else if constexpr (PART == 1) x = sv;
                    else if constexpr (PART == 2) x = qv - sv;
                    else x = qv * sv;
  #pragma unroll
                    for (int u = 0; u < 8; ++u) acc[a][u] = fmaf(x, w[u], acc[a][u]);
                  }
                }
              };
              run_part(std::integral_constant<int, 0>{});
              run_part(std::integral_constant<int, 1>{});
              run_part(std::integral_constant<int, 2>{});
              run_part(std::integral_constant<int, 3>{});
  #pragma unroll
              for (int a = 0; a < 4; ++a)
  #pragma unroll
                for (int u = 0; u < 8; ++u)
                  H1[(rg * 4 + a) * C::H1S + ug * 8 + u] = fmaxf(acc[a][u] + ms->b1[ug * 8 + u], 0.f);
            }
            __syncthreads();
            {
              // layer 2 + score: thread = 1 row x 8 units
              const int r = tid >> 3, u2 = tid & 7;
              float a2[8];
  #pragma unroll
              for (int u = 0; u < 8; ++u) a2[u] = 0.f;
              for (int k = 0; k < kN1; ++k) {
                const float h = H1[r * C::H1S + k];
                const float* wp = p.w2t + (long long)k * kN2 + u2 * 8;
                const float4 wa = __ldg(reinterpret_cast<const float4*>(wp));
                const float4 wb = __ldg(reinterpret_cast<const float4*>(wp + 4));
                a2[0] = fmaf(h, wa.x, a2[0]); a2[1] = fmaf(h, wa.y, a2[1]);
                a2[2] = fmaf(h, wa.z, a2[2]); a2[3] = fmaf(h, wa.w, a2[3]);
                a2[4] = fmaf(h, wb.x, a2[4]); a2[5] = fmaf(h, wb.y, a2[5]);
                a2[6] = fmaf(h, wb.z, a2[6]); a2[7] = fmaf(h, wb.w, a2[7]);
              }
              float part = 0.f;
  #pragma unroll
              for (int u = 0; u < 8; ++u) part += fmaxf(a2[u] + ms->b2[u2 * 8 + u], 0.f) * ms->w3[u2 * 8 + u];
              part += __shfl_xor_sync(0xffffffffu, part, 1);
              part += __shfl_xor_sync(0xffffffffu, part, 2);
              part += __shfl_xor_sync(0xffffffffu, part, 4);
              if (u2 == 0 && r < C::TM) ms->z[r] = part + b3;
            }
            __syncthreads();

          }
          softmax_tile(t0, n, tix, 0, false);
          if (has_next) seq_rows(nxt, min(C::TM, R - t1), 0);
        }
      }
    }
  }

  // ---------------------------------------------------------------- cleanup
  cp_async_wait_all();
  if constexpr (C::ATTN && C::MODE == 0) {
    if (tid == 0 && attn_ok && !weights_ready) {
      if (!mbar_wait(&ms->mbar_w, 0)) local_flags |= DSF_FLAG_TIMEOUT;
    }
    if (tid == 0 && ms->abort_ == 3) {
      // an MMA group did not complete in time: give it one more bounded wait
      // before the accumulator columns are released
      mbar_wait(&ms->mbar_mma, mma_phase ^ 1u);
      if constexpr (C::STREAM) {
        if (gk > 0) mbar_wait(&ms->mbar_done[(gk - 1u) % 3u], ((gk - 1u) / 3u) & 1u);
        for (uint32_t g = gk; g < gk + 2u; ++g) mbar_wait(&ms->mbar_full[g % 3u], (g / 3u) & 1u);
      }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      tc_fence_after();
      tmem_dealloc(ms->tmem_base, 512);
    }
  }
  if (tc_fail && tid == 0) local_flags |= DSF_FLAG_TIMEOUT;
  // one status write per warp
  local_flags = __reduce_or_sync(0xffffffffu, local_flags);
  if (lane == 0 && local_flags) flag(p.status, local_flags);
}

}  // namespace dsf
