// Backward of the sparse path and the sparse AdaGrad step (MultiTowerDIN:
// current state analysis, section 1 -- training with sparse AdaGrad -- and the
// forward of sections 4.2 and 4.4, differentiated).
//
// One call, in stream order:
//   scans      bag offsets of the KJT; raw and clamped sequence offsets
//   gather     per valid position: s (the three rows), x = [q, s, q-s, q*s]
//   GEMM 1, 2  recompute h1 = ReLU(x W1^T + b1), h2 pre-activation = h1 W2^T
//   softmax    per sample: z, a, da = ddin.s, dz = a (da - sum a da),
//              dh2 = dz w3 [h2 > 0], ds = a ddin; dw3, db2, db3
//   GEMM 3     dh1 pre-mask = dh2 W2;  mask [h1 > 0], db1
//   GEMM 4..6  dx = dh1 W1;  dW1 = dh1^T x;  dW2 = dh2^T h1
//   scatter    per sample: dq = sum_t (dx_q + dx_d + dx_p s_t), ds_t += dx_s -
//              dx_d + dx_p q; row gradients: ds_t slices into the sequence
//              rows, dpooled + dq slices into every value of the bags
// The six products are this library's GEMMs (gemm.cuh: tcgen05 with bf16
// operands, CUDA cores in the fp32 check mode), all in the A B^T form: the
// weights' transposes are packed per call, and the operands of the two
// weight gradients (sums over positions, split over K and reduced in order)
// are transposed into position-major rows. They run over the sequence
// values' length (rows past the valid count are zero).
// Row gradients are summed with vector fp32 atomics into caller-owned
// per-table buffers; the first contribution to a row appends it to a list,
// which the AdaGrad step walks.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "abi_checks.cuh"
#include "dinsparse.h"
#include "gemm.cuh"
#include "hash.cuh"
#include "launch.cuh"

namespace dsf {
namespace bwd {
namespace {

constexpr int kSplitCtas = 152;  // CTAs of the two weight-gradient products (K-splits x M-tiles)
constexpr int kRowBits = 40;
// The per-sample kernels (gather, softmax backward, dq/ds) take one warp per
// block: a block whose sample holds a long sequence then keeps only its own
// warp, and the freed warp slots take new blocks at once.
constexpr int kSampleWarps = 1, kSampleBlocks = 152 * 64;
constexpr int kScanThreads = 256, kScanRounds = 8, kScanTile = kScanThreads * kScanRounds;
constexpr int kMaxBlocks = 152 * 8;  // grid cap of the grid-stride kernels (their partial sums)
constexpr int kRedCols = 2 * 64 + 1;  // dw3 | db2 | db3 partials of the softmax kernel
constexpr int kRedChunks = 32;        // chunks of the column sums' first step
constexpr int kTile = 1024, kRowThreads = 512;  // row-gradient tiles (id occurrences) and their blocks
constexpr unsigned long long kNoKey = ~0ull;


size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// A second stream per device for the backward's steps that no next step
// needs (the KJT offsets, the weight packing, the bias-gradient columns).
// Work moves to it and back through events, so a graph capture of the call
// records the fork and the join. It is created by the first call that is not
// being captured (create false: only an existing one is returned). Null if
// it cannot be had: every step then runs on the call's stream.
cudaStream_t side_stream(int dev, bool create) {
  static std::mutex mu;
  static cudaStream_t cache[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev] && create && cudaStreamCreateWithFlags(&cache[dev], cudaStreamNonBlocking) != cudaSuccess) {
    cache[dev] = nullptr;
    (void)cudaGetLastError();
  }
  return cache[dev];
}
// `to` waits for everything enqueued on `from` so far.
bool follow(cudaStream_t to, cudaStream_t from) {
  if (to == from) return true;
  cudaEvent_t e;
  if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
  const bool ok = cudaEventRecord(e, from) == cudaSuccess && cudaStreamWaitEvent(to, e, 0) == cudaSuccess;
  cudaEventDestroy(e);  // (released once the record completes)
  return ok;
}

struct Layout {
  size_t boff, soff, roff, tsum, samp, zb, dab, part1, part2, gbag, okey, osrc, w1b, w2b, w1t, w2t, X, S, G1, H1, H2, dH2,
      dH1, dX, dS, XT, H1T, dH2T, dH1T, M1, split, red, total;
};

// Every buffer is sized for fp32 elements, so the layout does not depend on
// the MLP mode.
Layout layout(long long B, long long NV, long long Pc, int F, int D) {
  Layout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  const size_t Q = 3 * size_t(D), K1 = 12 * size_t(D), P = size_t(Pc);
  L.boff = take((size_t(F) * B + 1) * 8);
  L.soff = take((size_t(B) + 1) * 8);
  L.roff = take((size_t(B) + 1) * 8);
  L.tsum = take(4 * ((size_t(F) * B) / kScanTile + 2) * 8);
  L.samp = take(P * 4);
  L.zb = take(P * 4);
  L.dab = take(P * 4);
  L.part1 = take(size_t(kSampleBlocks) * kRedCols * 4);
  {
    // db1's partial sums: a row per block of the fp32 mask kernel, or four
    // per 128-position tile from the bf16 products' mask epilogue
    const size_t rows = size_t(4) * ((P + 127) / 128);
    L.part2 = take((rows > size_t(kMaxBlocks) ? rows : size_t(kMaxBlocks)) * kN1 * 4);
  }
  L.gbag = take(size_t(B) * F * D * 4);
  L.okey = take((size_t(NV) + 3 * P) * 8);
  L.osrc = take((size_t(NV) + 3 * P) * 8);
  L.w1b = take(size_t(kN1) * K1 * 2);
  L.w2b = take(size_t(kN2) * kN1 * 2);
  L.X = take(P * K1 * 4);
  L.S = take(P * Q * 4);
  L.G1 = take(P * kN1 * 4);
  L.H1 = take(P * kN1 * 4);
  L.H2 = take(P * kN2 * 4);
  L.dH2 = take(P * kN2 * 4);
  L.dH1 = take(P * kN1 * 4);
  L.dX = take(P * K1 * 4);
  L.dS = take(P * Q * 4);
  // transposed weights; transposed copies of x, h1, dh2, dh1 for the fp32
  // weight gradients (positions contiguous: rows of P8 = P rounded up to 8
  // elements, 16-byte aligned); split-K partials
  const size_t P8 = (P + 7) / 8 * 8;
  L.w1t = take(K1 * size_t(kN1) * 4);
  L.w2t = take(size_t(kN1) * kN2 * 4);
  L.XT = take(K1 * P8 * 4);
  L.H1T = take(size_t(kN1) * P8 * 4);
  L.dH2T = take(size_t(kN2) * P8 * 4);
  L.dH1T = take(size_t(kN1) * P8 * 4);
  L.M1 = take(P * (kN1 / 32) * 4);  // h1 > 0 as bits, one word per 32 columns
  {
    // one product alone (fp32) or both in one launch (bf16, kSplitCtas / 3 splits each)
    const size_t w1 = size_t(kSplitCtas / 2) * kN1 * K1, w2 = size_t(kSplitCtas) * kN2 * kN1;
    const size_t both = size_t(kSplitCtas / 3) * (size_t(kN1) * K1 + size_t(kN2) * kN1);
    const size_t m = w1 > w2 ? w1 : w2;
    L.split = take((m > both ? m : both) * 4);
  }
  L.red = take(size_t(kRedChunks) * (kRedCols + kN1) * 4);  // the column sums' chunk sums
  L.total = o;
  return L;
}

struct Params {
  const void* tables[kMaxF];
  long long rows[kMaxF];    // row count of the table's storage
  long long glimit[kMaxF];  // rows that are parameters (the hash pool's zero row is not)
  int sid[kMaxF];           // storage of table f (hash-table tables share one)
  float* grad[kMaxF];       // by storage
  int* touched[kMaxF];      // by storage
  unsigned int hash_mask;
  unsigned char kspace[kMaxF];
  const unsigned long long* hkeys;
  unsigned long long hbmask;
  int F, B, D, max_len;
  bool bf16_tables, bf16_mlp;
  unsigned int mean_mask;
  const long long* values;
  long long n_values;
  const long long* seq_values;
  long long n_seq;
  int q_feat[3], seq_table[3];
  long long* list;
  int* count;
  long long list_cap;
  int* status;
};

__device__ __forceinline__ long long rid(const Params& p, int f, long long id) {
  return ((p.hash_mask >> f) & 1u) ? hash::find(p.hkeys, p.hbmask, p.kspace[f], id) : id;
}

__device__ __forceinline__ void flag(int* status, int bits) {
  if (status && bits) atomicOr(status, bits);
}

// 16 table elements starting at element e of `row` (fp32 or bf16) as fp32
__device__ __forceinline__ void load16(const Params& p, const void* base, long long row, int e, float* v) {
  if (p.bf16_tables) {
    const uint4* q = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + row * p.D + e);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 w = __ldg(q + h);
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[h * 8 + 2 * i] = __uint_as_float(u[i] << 16);
        v[h * 8 + 2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
      }
    }
  } else {
    const float4* q = reinterpret_cast<const float4*>(static_cast<const float*>(base) + row * p.D + e);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float4 w = __ldg(q + h);
      v[4 * h] = w.x;
      v[4 * h + 1] = w.y;
      v[4 * h + 2] = w.z;
      v[4 * h + 3] = w.w;
    }
  }
}

// Records row `row` of storage s as touched (valid: the row is a parameter).
// The lanes that are first to touch a row reserve their list entries with
// one atomic per warp.
__device__ __forceinline__ int mark_row(const Params& p, int s, long long row, bool valid) {
  bool first = false;
  if (valid) {
    int* t = p.touched[s] + row;
    first = *reinterpret_cast<volatile int*>(t) == 0 && atomicExch(t, 1) == 0;
  }
  const unsigned act = __activemask();
  const unsigned want = __ballot_sync(act, first);
  if (!want) return 0;
  const int lane = threadIdx.x & 31, leader = __ffs(want) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(p.count, __popc(want));
  base = __shfl_sync(act, base, leader);
  if (!first) return 0;
  const int i = base + __popc(want & ((1u << lane) - 1u));
  if (i < p.list_cap) {
    p.list[i] = (static_cast<long long>(s) << kRowBits) | row;
    return 0;
  }
  return DSF_FLAG_GRAD_LIST;
}

// ---------------------------------------------------------------- kernels
// Block-wide inclusive scan of two 64-bit values (256 threads); returns the
// block totals through the references.
__device__ __forceinline__ void block_scan2(long long& a, long long& b, long long& ta, long long& tb) {
  __shared__ long long wa[kScanThreads / 32], wb[kScanThreads / 32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o);
    if (lane >= o) a += ya, b += yb;
  }
  if (lane == 31) wa[w] = a, wb[w] = b;
  __syncthreads();
  long long pa = 0, pb = 0;
  ta = tb = 0;
#pragma unroll
  for (int i = 0; i < kScanThreads / 32; ++i) {
    if (i < w) pa += wa[i], pb += wb[i];
    ta += wa[i], tb += wb[i];
  }
  a += pa;
  b += pb;
  __syncthreads();
}

// One scan: the exclusive scans of max(len, 0) (raw) and, when clp is given,
// of min(max(len, 0), clamp) over n entries, in tiles of kScanTile.
struct ScanJob {
  const int* len;
  int n, clamp, tiles;
  long long *tsum, *raw, *clp;
};
// Both scans of a call run in the same two launches: blocks [0, tiles of job
// 0) take job 0, the rest job 1.
struct ScanJobs {
  ScanJob j[2];
};
__device__ __forceinline__ const ScanJob& job_of(const ScanJobs& J, int& tile) {
  const int which = int(blockIdx.x) < J.j[0].tiles ? 0 : 1;
  tile = int(blockIdx.x) - (which ? J.j[0].tiles : 0);
  return J.j[which];
}

// Pass 1: the sums of each tile (coalesced loads).
__global__ void __launch_bounds__(kScanThreads) scan_tiles_kernel(const ScanJobs jobs) {
  int tile;
  const ScanJob& J = job_of(jobs, tile);
  long long a = 0, b = 0;
  for (int r = 0; r < kScanRounds; ++r) {
    const long long k = (long long)tile * kScanTile + r * kScanThreads + threadIdx.x;
    if (k < J.n) {
      const int v = max(J.len[k], 0);
      a += v;
      b += min(v, J.clamp);
    }
  }
  long long ta, tb;
  block_scan2(a, b, ta, tb);
  if (threadIdx.x == 0) J.tsum[2 * tile] = ta, J.tsum[2 * tile + 1] = tb;
}

// Pass 2: each tile adds the sums of the tiles before it and scans its own
// entries, kScanRounds consecutive ones per thread (one block scan of the
// threads' sums); the last tile writes the totals at index n.
__global__ void __launch_bounds__(kScanThreads) scan_apply_kernel(const ScanJobs jobs) {
  int tile;
  const ScanJob& J = job_of(jobs, tile);
  long long ca = 0, cb = 0;
  for (int i = threadIdx.x; i < tile; i += kScanThreads) ca += J.tsum[2 * i], cb += J.tsum[2 * i + 1];
  {
    long long ta, tb;
    block_scan2(ca, cb, ta, tb);
    ca = ta, cb = tb;
  }
  const long long k0 = (long long)tile * kScanTile + (long long)threadIdx.x * kScanRounds;
  int v[kScanRounds];
  long long a = 0, b = 0;
#pragma unroll
  for (int r = 0; r < kScanRounds; ++r) {
    v[r] = k0 + r < J.n ? max(J.len[k0 + r], 0) : 0;
    a += v[r];
    b += min(v[r], J.clamp);
  }
  const long long own_a = a, own_b = b;
  long long ta, tb;
  block_scan2(a, b, ta, tb);
  long long ea = ca + a - own_a, eb = cb + b - own_b;  // the exclusive prefix at entry k0
#pragma unroll
  for (int r = 0; r < kScanRounds; ++r) {
    if (k0 + r < J.n) {
      J.raw[k0 + r] = ea;
      if (J.clp) J.clp[k0 + r] = eb;
    }
    ea += v[r];
    eb += min(v[r], J.clamp);
  }
  if (tile == J.tiles - 1 && threadIdx.x == 0) {
    J.raw[J.n] = ca + ta;
    if (J.clp) J.clp[J.n] = cb + tb;
  }
}

// Column sums over the rows of [rows, cols] fp32 partial-sum arrays, in a
// fixed order: part0 ([rows0, kRedCols]) into dw3 | db2 | db3 and, when given,
// part1 ([rows1, kN1]) into db1. Two steps: chunk sums (reduce_chunks_kernel)
// and then one block per column over the chunks (reduce_cols_kernel).
struct RedJobs {
  const float* part0;
  int rows0;
  const float* part1;
  int rows1;
  float *dw3, *db2, *db3, *db1;
};
// Step 1: block (group g, chunk k) sums 32 columns of rows [k rows / 32,
// (k + 1) rows / 32), eight rows at a time (each warp reads a row's 128
// bytes), and writes the chunk's sums to row k of out0 (part0's columns) or
// out1 (part1's). Blocks [0, 5) x 32 take part0, the rest part1.
__global__ void __launch_bounds__(256) reduce_chunks_kernel(const RedJobs r, float* __restrict__ out0,
                                                             float* __restrict__ out1) {
  constexpr int G0 = (kRedCols + 31) / 32;
  __shared__ float sh[8][33];
  const bool first = int(blockIdx.x) < G0;
  const int g = first ? int(blockIdx.x) : int(blockIdx.x) - G0;
  const float* part = first ? r.part0 : r.part1;
  const int rows = first ? r.rows0 : r.rows1, cols = first ? kRedCols : kN1;
  float* out = first ? out0 : out1;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5, c = g * 32 + tx, k = blockIdx.y;
  const long long r0 = (long long)rows * k / kRedChunks, r1 = (long long)rows * (k + 1) / kRedChunks;
  float v = 0.f;
  if (c < cols) {
#pragma unroll 8
    for (long long i = r0 + ty; i < r1; i += 8) v += part[i * cols + c];
  }
  sh[ty][tx] = v;
  __syncthreads();
  if (ty == 0 && c < cols) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += sh[w][tx];
    out[(long long)k * cols + c] = t;
  }
}
__global__ void __launch_bounds__(256) reduce_cols_kernel(const RedJobs r) {
  __shared__ float sh[256];
  const bool first = int(blockIdx.x) < kRedCols;
  const int c = first ? int(blockIdx.x) : int(blockIdx.x) - kRedCols;
  const float* part = first ? r.part0 : r.part1;
  const int rows = first ? r.rows0 : r.rows1, cols = first ? kRedCols : kN1;
  float v = 0.f;
  for (int i = threadIdx.x; i < rows; i += 256) v += part[(long long)i * cols + c];
  sh[threadIdx.x] = v;
  __syncthreads();
  for (int o = 128; o; o >>= 1) {
    if (threadIdx.x < o) sh[threadIdx.x] += sh[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (!first) r.db1[c] = sh[0];
    else if (c < kN2) r.dw3[c] = sh[0];
    else if (c < 2 * kN2) r.db2[c - kN2] = sh[0];
    else r.db3[0] = sh[0];
  }
}


template <class T>
__device__ __forceinline__ void store4(T* dst, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<float>(float* dst, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(dst) = make_float4(a, b, c, d);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, float a, float b, float c, float d) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&lo);
  u.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(dst) = u;
}
// 8 consecutive elements (16-byte aligned for bf16: one 16-byte store)
template <class T>
__device__ __forceinline__ void store8(T* dst, const float* v);
template <>
__device__ __forceinline__ void store8<float>(float* dst, const float* v) {
  *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(dst + 4) = make_float4(v[4], v[5], v[6], v[7]);
}
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* dst, const float* v) {
  uint32_t u[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    u[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(dst) = make_uint4(u[0], u[1], u[2], u[3]);
}

// One warp per sample, one lane per position: its sample, s (fp32), x =
// [q, s, q - s, q * s] (the MLP operand type) and the occurrence keys of its
// three sequence ids. Rows past the valid count are zeroed.
template <class T>
__global__ void __launch_bounds__(kSampleWarps * 32, 32 / kSampleWarps) gather_kernel(
    const Params p, const float* __restrict__ pooled, const long long* __restrict__ soff,
    const long long* __restrict__ roff, int* samp, T* X, float* S, long long Pc, unsigned long long* __restrict__ okey,
    long long* __restrict__ osrc) {
  const int D = p.D, Q = 3 * D, K1 = 4 * Q, FD = p.F * D;
  const int lane = threadIdx.x & 31;
  const long long P = min(soff[p.B], Pc);
  int flags = (soff[p.B] > Pc && blockIdx.x == 0 && threadIdx.x == 0) ? DSF_FLAG_COUNT : 0;
  const int nwarps = gridDim.x * kSampleWarps;
  for (int b = blockIdx.x * kSampleWarps + (threadIdx.x >> 5); b < p.B; b += nwarps) {
    const long long p0 = min(soff[b], Pc), p1 = min(soff[b + 1], Pc);
    for (long long pos = p0 + lane; pos < p1; pos += 32) {
      T* x = X + pos * K1;
      samp[pos] = b;
      const long long j = roff[b] + (pos - soff[b]);
      long long row[3];
      bool ok[3];
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        const int tb = p.seq_table[k];
        long long id = -1;
        if (j < p.n_seq) id = rid(p, tb, p.seq_values[k * p.n_seq + j]);
        else flags |= DSF_FLAG_COUNT;
        ok[k] = id >= 0 && id < p.rows[tb];
        if (!ok[k] && j < p.n_seq) flags |= DSF_FLAG_ID_RANGE;
        row[k] = ok[k] ? id : 0;
        // the occurrence of this sequence id (its gradient is row 3 pos + k
        // of ds): storage << 40 | row, or none
        const long long o = p.n_values + 3 * pos + k;
        okey[o] = (id >= 0 && id < p.glimit[tb])
                      ? (static_cast<unsigned long long>(p.sid[tb]) << kRowBits) | static_cast<unsigned long long>(id)
                      : kNoKey;
        osrc[o] = -(3 * pos + k) - 1;
      }
      for (int c = 0; c < Q / 16; ++c) {
        const int k = (c * 16) / D, e = (c * 16) % D;
        float sv[16], q[16];
        if (ok[k]) load16(p, p.tables[p.seq_table[k]], row[k], e, sv);
        else
#pragma unroll
          for (int i = 0; i < 16; ++i) sv[i] = 0.f;
        const float4* qp = reinterpret_cast<const float4*>(pooled + (long long)b * FD + p.q_feat[k] * D + e);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float4 v = __ldg(qp + h);
          q[4 * h] = v.x, q[4 * h + 1] = v.y, q[4 * h + 2] = v.z, q[4 * h + 3] = v.w;
        }
        float* sd = S + pos * Q + c * 16;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int i = 4 * h;
          *reinterpret_cast<float4*>(sd + i) = make_float4(sv[i], sv[i + 1], sv[i + 2], sv[i + 3]);
        }
        // x's four parts, eight elements per store
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = 8 * h;
          float dq[8], pq[8];
#pragma unroll
          for (int t = 0; t < 8; ++t) dq[t] = q[i + t] - sv[i + t], pq[t] = q[i + t] * sv[i + t];
          store8<T>(x + c * 16 + i, q + i);
          store8<T>(x + Q + c * 16 + i, sv + i);
          store8<T>(x + 2 * Q + c * 16 + i, dq);
          store8<T>(x + 3 * Q + c * 16 + i, pq);
        }
      }
    }
  }
  for (long long i = P * K1 / 4 + blockIdx.x * (long long)blockDim.x + threadIdx.x; i < Pc * K1 / 4;
       i += (long long)gridDim.x * blockDim.x)
    store4<T>(X + 4 * i, 0.f, 0.f, 0.f, 0.f);
  flag(p.status, flags);
}

// h1 = ReLU(G1 + b1) in the MLP operand type, over [Pc, 256] (the fp32 check
// mode; bf16 mode does it in the product's epilogue).
template <class T>
__global__ void relu1_kernel(const float* __restrict__ G1, const float* __restrict__ b1, T* H1, long long n4) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    const float4 g = reinterpret_cast<const float4*>(G1)[i];
    const int c = int((i * 4) % kN1);
    store4<T>(H1 + i * 4, fmaxf(g.x + b1[c], 0.f), fmaxf(g.y + b1[c + 1], 0.f), fmaxf(g.z + b1[c + 2], 0.f),
              fmaxf(g.w + b1[c + 3], 0.f));
  }
}

template <class T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }

template <class T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// The MLP weights as the products read them: W1 [256, K1] and W2 [64, 256]
// as given, and their transposes W1^T [K1, 256], W2^T [256, 64], in the
// operand type T (bf16: rounded to nearest even). perm: W1^T's row for
// column g Q + d of x (part g of cat[q, s, q - s, q s], dim d) is 4 d + g,
// so that the dx product's columns come four per dim (the dq/ds epilogue).
template <class T>
__global__ void pack_kernel(const float* __restrict__ W1, const float* __restrict__ W2, int K1, T* w1, T* w2,
                            T* w1t, T* w2t, bool perm) {
  const int n1 = kN1 * K1, n2 = kN2 * kN1, Q = K1 / 4;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n1 + n2; i += gridDim.x * blockDim.x) {
    if (i < n1) {
      const int o = i / K1, k = i - o * K1;
      const T v = from_f<T>(W1[i]);
      if (w1) w1[i] = v;
      const int r = perm ? 4 * (k % Q) + k / Q : k;
      w1t[(long long)r * kN1 + o] = v;
    } else {
      const int j = i - n1, o = j / kN1, k = j - o * kN1;
      const T v = from_f<T>(W2[j]);
      if (w2) w2[j] = v;
      w2t[(long long)k * kN2 + o] = v;
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp per sample (and per block, as in the gather): softmax and score
// backward over the sample's positions. z and da = ddin.s take one lane per
// position; dH2, dS and the sums of dw3, db2, db3 take one position per step
// with the lanes over dimensions (steps are independent). Writes each
// block's partial sums (dw3 | db2 | db3) as a row; rows of dH2 past the valid
// count are zeroed.
template <class T>
__global__ void __launch_bounds__(32, 32) softmax_bwd_kernel(
    const Params p, const long long* __restrict__ soff, const float* __restrict__ H2, const float* __restrict__ S,
    const float* __restrict__ ddin, const float* __restrict__ b2, const float* __restrict__ w3,
    const float* __restrict__ b3, float* __restrict__ zb, float* __restrict__ dab, T* __restrict__ dH2,
    float* __restrict__ dS, float* __restrict__ part, long long Pc) {
  __shared__ float sw3[kN2], sb2[kN2];
  const int lane = threadIdx.x;
  const int Q = 3 * p.D;
  for (int i = lane; i < kN2; i += 32) sw3[i] = w3[i], sb2[i] = b2[i];
  __syncwarp();
  const float bb3 = __ldg(b3);
  float acc_w3[2] = {0.f, 0.f}, acc_b2[2] = {0.f, 0.f}, acc_b3 = 0.f;
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    const long long p0 = min(soff[b], Pc), p1 = min(soff[b + 1], Pc);
    if (p1 <= p0) continue;
    const float* dd = ddin + (long long)b * Q;
    // z and da per position (a lane each), the running max
    float m = -INFINITY;
    for (long long q = p0 + lane; q < p1; q += 32) {
      const float4* h = reinterpret_cast<const float4*>(H2 + q * kN2);
      float z = bb3;
#pragma unroll 4
      for (int i = 0; i < kN2 / 4; ++i) {
        const float4 v = h[i];
        z += sw3[4 * i] * fmaxf(v.x + sb2[4 * i], 0.f) + sw3[4 * i + 1] * fmaxf(v.y + sb2[4 * i + 1], 0.f) +
             sw3[4 * i + 2] * fmaxf(v.z + sb2[4 * i + 2], 0.f) + sw3[4 * i + 3] * fmaxf(v.w + sb2[4 * i + 3], 0.f);
      }
      const float4* sr = reinterpret_cast<const float4*>(S + q * Q);
      const float4* dr = reinterpret_cast<const float4*>(dd);
      float da = 0.f;
      for (int i = 0; i < Q / 4; ++i) {
        const float4 x = sr[i], y = __ldg(dr + i);
        da += x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
      }
      zb[q] = z;
      dab[q] = da;
      m = fmaxf(m, z);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f, sda = 0.f;
    for (long long q = p0 + lane; q < p1; q += 32) {
      const float e = expf(zb[q] - m);
      l += e;
      sda += e * dab[q];
      zb[q] = e;
    }
    l = warp_sum(l);
    sda = warp_sum(sda);
    const float c = sda / l, il = 1.f / l;
    // each lane's a and dz for its positions, handed out one position per step
    for (long long q0 = p0; q0 < p1; q0 += 32) {
      const long long qm = q0 + lane;
      float a_l = 0.f, dz_l = 0.f;
      if (qm < p1) {
        a_l = zb[qm] * il;
        dz_l = a_l * (dab[qm] - c);
      }
      const int n = int(min((long long)32, p1 - q0));
#pragma unroll 4
      for (int t = 0; t < n; ++t) {
        const long long q = q0 + t;
        const float a = __shfl_sync(0xffffffffu, a_l, t), dz = __shfl_sync(0xffffffffu, dz_l, t);
        const float pa = H2[q * kN2 + lane] + sb2[lane], pb = H2[q * kN2 + lane + 32] + sb2[lane + 32];
        const float ga = pa > 0.f ? dz * sw3[lane] : 0.f, gb = pb > 0.f ? dz * sw3[lane + 32] : 0.f;
        dH2[q * kN2 + lane] = from_f<T>(ga);
        dH2[q * kN2 + lane + 32] = from_f<T>(gb);
        acc_w3[0] += dz * fmaxf(pa, 0.f);
        acc_w3[1] += dz * fmaxf(pb, 0.f);
        acc_b2[0] += ga;
        acc_b2[1] += gb;
        if (lane == 0) acc_b3 += dz;
        for (int d = lane; d < Q; d += 32) dS[q * Q + d] = a * dd[d];
      }
    }
  }
  float* row = part + (long long)blockIdx.x * kRedCols;
  row[lane] = acc_w3[0];
  row[lane + 32] = acc_w3[1];
  row[lane + 64] = acc_b2[0];
  row[lane + 96] = acc_b2[1];
  if (lane == 0) row[2 * kN2] = acc_b3;
  // rows past the valid count: zero gradient
  const long long P = min(soff[p.B], Pc);
  for (long long i = P * kN2 + blockIdx.x * (long long)blockDim.x + threadIdx.x; i < Pc * kN2;
       i += (long long)gridDim.x * blockDim.x)
    dH2[i] = from_f<T>(0.f);
}

// dh1 = G (dh2 W2) * [h1 > 0], over [Pc, 256] with one column per thread;
// db1 sums the masked values (the fp32 check mode; bf16 mode does it in the
// product's epilogue).
template <class T>
__global__ void __launch_bounds__(kN1) relu1_bwd_kernel(const float* __restrict__ G, const T* __restrict__ H1,
                                                       T* dH1, float* part, long long Pc) {
  const int c = threadIdx.x;
  float acc = 0.f;
  for (long long r = blockIdx.x; r < Pc; r += gridDim.x) {
    const long long i = r * kN1 + c;
    const float v = to_f<T>(H1[i]) > 0.f ? G[i] : 0.f;
    dH1[i] = from_f<T>(v);
    acc += v;
  }
  part[(long long)blockIdx.x * kN1 + c] = acc;
}

__device__ __forceinline__ float4 f4(const float* q) { return *reinterpret_cast<const float4*>(q); }
__device__ __forceinline__ float4 operator+(float4 a, float4 b) { return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }
__device__ __forceinline__ float4 operator-(float4 a, float4 b) { return make_float4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w); }
__device__ __forceinline__ float4 operator*(float4 a, float4 b) { return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w); }
__device__ __forceinline__ float4 scale4(float4 a, float s) { return make_float4(a.x * s, a.y * s, a.z * s, a.w * s); }

// One warp per sample, no atomics. Positions, a lane each: the final ds =
// dS + dx_s - dx_d + dx_p q (in place) and the lane's share of dq = sum_t
// (dx_q + dx_d + dx_p s_t), reduced over the lanes afterwards. Then the bags,
// one (feature, 4-element piece) per lane step: g = dpooled + dq (over L for
// mean pooling) into the bag-gradient rows. Pieces of x are handled kPG at a
// time so the dq shares stay in registers. (The occurrence keys come from the
// gather and from kjt_keys_kernel.)
constexpr int kPG = 4;
__global__ void __launch_bounds__(kSampleWarps * 32, 32 / kSampleWarps) dsdq_kernel(
    const Params p, const long long* __restrict__ boff, const long long* __restrict__ soff,
    const long long* __restrict__ roff, long long Pc, const float* __restrict__ pooled,
    const float* __restrict__ dpooled, const float* __restrict__ dX, const float* __restrict__ S,
    float* __restrict__ dS, float* __restrict__ gbag, const float* __restrict__ dqc) {
  __shared__ float dqs[kSampleWarps][3 * 64];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int D = p.D, Q = 3 * D, K1 = 4 * Q, FD = p.F * D, nc = Q / 4;
  int flags = 0;
  for (int b = blockIdx.x * kSampleWarps + warp; b < p.B; b += gridDim.x * kSampleWarps) {
    const long long p0 = min(soff[b], Pc), p1 = min(soff[b + 1], Pc);
    const float* qrow = pooled + (long long)b * FD;
    for (int g0 = 0; g0 < nc; g0 += kPG) {
      float4 dq[kPG];
#pragma unroll
      for (int i = 0; i < kPG; ++i) dq[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (long long q = p0 + lane; q < p1; q += 32) {
        if (dqc) {  // (ds and the dq terms came from the dx product's epilogue)
#pragma unroll
          for (int i = 0; i < kPG; ++i)
            if (g0 + i < nc) dq[i] = dq[i] + f4(dqc + q * Q + 4 * (g0 + i));
          continue;
        }
        const float* dx = dX + q * K1;
#pragma unroll
        for (int i = 0; i < kPG; ++i) {
          const int c4 = g0 + i;
          if (c4 >= nc) break;
          const int d = 4 * c4, k = d / D, e = d % D;
          const float4 xq = f4(dx + d), xs = f4(dx + Q + d), xd = f4(dx + 2 * Q + d), xp = f4(dx + 3 * Q + d);
          const float4 s4 = f4(S + q * Q + d);
          const float4 q4 = f4(qrow + p.q_feat[k] * D + e);
          dq[i] = dq[i] + xq + xd + xp * s4;
          float* dsp = dS + q * Q + d;
          *reinterpret_cast<float4*>(dsp) = f4(dsp) + xs - xd + xp * q4;
        }
      }
#pragma unroll
      for (int i = 0; i < kPG; ++i) {
        float4 v = dq[i];
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
          v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
          v.z += __shfl_xor_sync(0xffffffffu, v.z, o);
          v.w += __shfl_xor_sync(0xffffffffu, v.w, o);
        }
        if (lane == 0 && g0 + i < nc) *reinterpret_cast<float4*>(&dqs[warp][4 * (g0 + i)]) = v;
      }
    }
    __syncwarp();
    const int npieces = p.F * (D / 4);
    for (int c = lane; c < npieces; c += 32) {
      const int f = c / (D / 4), e = (c % (D / 4)) * 4;
      float4 g = dpooled ? f4(dpooled + (long long)b * FD + f * D + e) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 3; ++k)
        if (p.q_feat[k] == f) g = g + *reinterpret_cast<const float4*>(&dqs[warp][k * D + e]);
      const long long v0 = boff[(long long)f * p.B + b], v1 = boff[(long long)f * p.B + b + 1];
      if (v1 > v0 && ((p.mean_mask >> f) & 1u)) g = scale4(g, 1.f / float(v1 - v0));
      *reinterpret_cast<float4*>(gbag + (long long)b * FD + f * D + e) = g;
    }
    __syncwarp();
  }
  flag(p.status, flags);
}

// The occurrences of the KJT's values, one thread per bag: value v of bag
// (f, b) gets the key storage << 40 | row (or none) and its gradient row
// b F + f of the bag gradients.
__global__ void __launch_bounds__(256) kjt_keys_kernel(const Params p, const long long* __restrict__ boff,
                                                       unsigned long long* __restrict__ okey,
                                                       long long* __restrict__ osrc) {
  int flags = 0;
  const long long nb = (long long)p.F * p.B;
  for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < nb; g += (long long)gridDim.x * blockDim.x) {
    const int f = int(g / p.B);
    const long long b = g - (long long)f * p.B;
    const long long v0 = boff[g], v1 = boff[g + 1];
    for (long long v = v0; v < v1; ++v) {
      if (v >= p.n_values) {
        flags |= DSF_FLAG_COUNT;
        break;
      }
      const long long id = rid(p, f, p.values[v]);
      okey[v] = (id >= 0 && id < p.glimit[f])
                    ? (static_cast<unsigned long long>(p.sid[f]) << kRowBits) | static_cast<unsigned long long>(id)
                    : kNoKey;
      osrc[v] = b * p.F + f;
    }
  }
  flag(p.status, flags);
}

__device__ __forceinline__ float4 shfl_up4(float4 v, int o) {
  return make_float4(__shfl_up_sync(0xffffffffu, v.x, o), __shfl_up_sync(0xffffffffu, v.y, o),
                     __shfl_up_sync(0xffffffffu, v.z, o), __shfl_up_sync(0xffffffffu, v.w, o));
}

// Row gradients of a tile of kTile id occurrences (the KJT's values at
// [0, n_values), the sequence ids at n_values + 3 * position + k): the tile's
// keys sorted with their tile indices (bitonic network, two elements per
// thread: registers, shuffles, and shared memory only for distances of 64
// and more), then
// per 4-element piece a segmented inclusive scan over the sorted order (two
// elements per thread, shuffles within warps, a carry across warps) gives each
// run's sum at its last element, which issues one vector reduction into the
// row's gradient (the first piece also marks the row touched). Occurrences
// past the valid counts or with no parameter row sort last and are skipped.
__global__ void __launch_bounds__(kRowThreads) rowgrad_kernel(
    const Params p, const long long* __restrict__ boff, const long long* __restrict__ soff, long long Pc,
    const unsigned long long* __restrict__ okey, const long long* __restrict__ osrc, const float* __restrict__ gbag,
    const float* __restrict__ dS) {
  constexpr int NW = kRowThreads / 32;
  static_assert(kTile == 2 * kRowThreads && kTile <= 1024, "two elements per thread; tile index in 10 bits");
  __shared__ unsigned long long key[kTile];
  __shared__ long long src[kTile];
  __shared__ uint16_t sidx[kTile];
  __shared__ float4 wagg[NW];
  __shared__ int whead[NW];
  const int D = p.D, Q = 3 * D, pieces = D / 4, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const long long nv = min(boff[(long long)p.F * p.B], p.n_values), P = min(soff[p.B], Pc);
  const long long o0 = (long long)blockIdx.x * kTile;
  // sort words: key << 10 | tile index (keys hold at most 45 bits; an
  // occurrence with no parameter row sorts last as all ones). Equal keys
  // keep their occurrence order, so each run is summed in that order.
  unsigned long long v[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int i = 2 * tid + e;
    const long long o = o0 + i;
    const bool ok = o < p.n_values ? o < nv : (o - p.n_values) < 3 * P;
    const unsigned long long k = ok ? okey[o] : kNoKey;
    src[i] = ok ? osrc[o] : 0;
    v[e] = k == kNoKey ? ~0ull : (k << 10) | unsigned(i);
  }
  // bitonic network over positions 2 tid + e: distance 1 within the thread,
  // 2 .. 32 across lanes (shuffles), 64 and up through shared memory
  for (int k = 2; k <= kTile; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      unsigned long long q[2];
      if (j == 1) {
        q[0] = v[1];
        q[1] = v[0];
      } else if (j <= 32) {
#pragma unroll
        for (int e = 0; e < 2; ++e) q[e] = __shfl_xor_sync(0xffffffffu, v[e], j >> 1);
      } else {
        __syncthreads();  // (the previous stage's reads are done)
        key[2 * tid] = v[0];
        key[2 * tid + 1] = v[1];
        __syncthreads();
#pragma unroll
        for (int e = 0; e < 2; ++e) q[e] = key[(2 * tid + e) ^ j];
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int i = 2 * tid + e;
        const bool up = (i & k) == 0, low = (i & j) == 0;
        const unsigned long long lo = v[e] < q[e] ? v[e] : q[e], hi = v[e] < q[e] ? q[e] : v[e];
        v[e] = (low == up) ? lo : hi;
      }
    }
  }
  __syncthreads();  // (the last shared-memory stage's reads are done)
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    key[2 * tid + e] = v[e] == ~0ull ? kNoKey : v[e] >> 10;
    sidx[2 * tid + e] = uint16_t(v[e] & 1023u);
  }
  __syncthreads();
  const int ia = 2 * tid, ib = ia + 1;
  const unsigned long long ka = key[ia], kb = key[ib];
  const unsigned long long kn = ib + 1 < kTile ? key[ib + 1] : kNoKey;
  const bool va = ka != kNoKey, vb = kb != kNoKey;
  const bool sa = va && (ia == 0 || key[ia - 1] != ka), sb = vb && ka != kb;
  const bool ea = va && ka != kb, eb = vb && kn != kb;  // last element of a run
  auto piece = [&](long long sj, int c) {
    const float* v = sj >= 0 ? gbag + sj * D : dS + ((-sj - 1) / 3) * Q + ((-sj - 1) % 3) * D;
    return f4(v + 4 * c);
  };
  int flags = 0;
  for (int c = 0; c < pieces; ++c) {
    const float4 xa = va ? piece(src[sidx[ia]], c) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 xb = vb ? piece(src[sidx[ib]], c) : make_float4(0.f, 0.f, 0.f, 0.f);
    // this thread's trailing segment (from its last run start, or all of it)
    float4 agg = sb ? xb : xa + xb;
    bool head = sa || sb;
    // segmented inclusive scan over the warp's lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float4 y = shfl_up4(agg, o);
      const bool hy = __shfl_up_sync(0xffffffffu, head, o);
      if (lane >= o) {
        if (!head) agg = agg + y;
        head = head || hy;
      }
    }
    if (lane == 31) wagg[w] = agg, whead[w] = head;
    __syncthreads();
    // the carry into this warp: the trailing segments of the warps before it
    float4 cw = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int u = w - 1; u >= 0; --u) {
      cw = cw + wagg[u];
      if (whead[u]) break;
    }
    // the carry into this thread's first element
    const float4 prev = shfl_up4(agg, 1);
    const bool hprev = __shfl_up_sync(0xffffffffu, head, 1);
    float4 carry = lane == 0 ? cw : (hprev ? prev : prev + cw);
    const float4 ta = sa ? xa : carry + xa;  // run sums through element a and b
    const float4 tb = sb ? xb : ta + xb;
    const float4 tot[2] = {ta, tb};
    const bool end[2] = {ea, eb};
    const unsigned long long kk[2] = {ka, kb};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int s = int(kk[h] >> kRowBits);
      const long long row = end[h] ? (long long)(kk[h] & ((1ull << kRowBits) - 1)) : 0;
      if (end[h]) {
        float* dst = p.grad[s] + row * D + 4 * c;
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(tot[h].x), "f"(tot[h].y),
                     "f"(tot[h].z), "f"(tot[h].w)
                     : "memory");
      }
      if (c == 0) flags |= mark_row(p, end[h] ? s : 0, row, end[h]);
    }
    __syncthreads();
  }
  flag(p.status, flags);
}

struct Upd {
  void* table[kMaxF];
  float* accum[kMaxF];
  float* grad[kMaxF];
  int* touched[kMaxF];
  const long long* list;
  const int* count;
  long long cap;
  int D;
  float lr, eps;
};

// AdaGrad over the touched rows (4 elements per thread), then the row's
// gradient and touched flag are cleared.
template <bool BF16>
__global__ void update_kernel(const Upd u) {
  const long long n = min((long long)*u.count, u.cap);
  const int pieces = u.D / 4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n * pieces;
       i += (long long)gridDim.x * blockDim.x) {
    const long long ent = u.list[i / pieces];
    const int s = int(ent >> kRowBits), e = int(i % pieces) * 4;
    const long long row = ent & ((1ll << kRowBits) - 1);
    float* gp = u.grad[s] + row * u.D + e;
    float* Gp = u.accum[s] + row * u.D + e;
    const float4 g = *reinterpret_cast<float4*>(gp);
    float4 G = *reinterpret_cast<float4*>(Gp);
    G.x += g.x * g.x, G.y += g.y * g.y, G.z += g.z * g.z, G.w += g.w * g.w;
    *reinterpret_cast<float4*>(Gp) = G;
    const float dw[4] = {u.lr * g.x / (sqrtf(G.x) + u.eps), u.lr * g.y / (sqrtf(G.y) + u.eps),
                         u.lr * g.z / (sqrtf(G.z) + u.eps), u.lr * g.w / (sqrtf(G.w) + u.eps)};
    if (BF16) {
      __nv_bfloat16* w = static_cast<__nv_bfloat16*>(u.table[s]) + row * u.D + e;
#pragma unroll
      for (int k = 0; k < 4; ++k) w[k] = __float2bfloat16_rn(__bfloat162float(w[k]) - dw[k]);
    } else {
      float4* w = reinterpret_cast<float4*>(static_cast<float*>(u.table[s]) + row * u.D + e);
      float4 v = *w;
      v.x -= dw[0], v.y -= dw[1], v.z -= dw[2], v.w -= dw[3];
      *w = v;
    }
    *reinterpret_cast<float4*>(gp) = make_float4(0.f, 0.f, 0.f, 0.f);
    if (e == 0) u.touched[s][row] = 0;
  }
}

__global__ void reset_count_kernel(int* count) { *count = 0; }

// ---------------------------------------------------------------- host
int grid_for(long long n, int threads, int cap = 152 * 16) {
  long long g = (n + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > cap) g = cap;
  return int(g);
}

// The column sums of the partial-sum arrays (two launches on st; red holds
// the chunk sums).
bool col_sums(const RedJobs& r, float* red, cudaStream_t st) {
  float *out0 = red, *out1 = red + size_t(kRedChunks) * kRedCols;
  const int g = (kRedCols + 31) / 32 + (r.part1 ? kN1 / 32 : 0);
  reduce_chunks_kernel<<<dim3(g, kRedChunks), 256, 0, st>>>(r, out0, out1);
  RedJobs c = r;
  c.part0 = out0;
  c.rows0 = kRedChunks;
  if (r.part1) c.part1 = out1, c.rows1 = kRedChunks;
  reduce_cols_kernel<<<kRedCols + (r.part1 ? kN1 : 0), 256, 0, st>>>(c);
  return cudaGetLastError() == cudaSuccess;
}

// Storage of table f: hash-table tables share the first such table's index.
int storage_of(const dsf_tables* t, int f) {
  if (!hashed(t, f)) return f;
  for (int g = 0; g < t->F; ++g)
    if (hashed(t, g)) return g;
  return f;
}

int check_row_state(const dsf_tables* t, float* const* grad, int32_t* const* touched) {
  for (int f = 0; f < t->F; ++f) {
    const int s = storage_of(t, f);
    if (!grad[f] || !aligned(grad[f], 16) || (touched && !touched[f])) return DSF_EINVAL;
    if (s != f && (grad[f] != grad[s] || (touched && touched[f] != touched[s]))) return DSF_EINVAL;
  }
  return DSF_OK;
}

void fill_tables(Params& p, const dsf_tables* t) {
  hash::Layout L{};
  uint8_t* hw = nullptr;
  if (t->hash) {
    L = hash::layout(t->hash->capacity, t->hash->D, t->dtype == DSF_BF16 ? 2 : 4);
    hw = static_cast<uint8_t*>(t->hash->workspace);
    p.hkeys = reinterpret_cast<const unsigned long long*>(hw + L.keys_off);
    p.hbmask = L.n_buckets - 1;
  }
  for (int f = 0; f < t->F; ++f) {
    if (hashed(t, f)) {
      p.tables[f] = hw + L.pool_off;
      p.rows[f] = static_cast<long long>(L.n_slots) + 1;
      p.glimit[f] = static_cast<long long>(L.n_slots);
      p.hash_mask |= 1u << f;
      p.kspace[f] = static_cast<unsigned char>(t->hash->key_space[f]);
    } else {
      p.tables[f] = t->table_ptrs[f];
      p.rows[f] = p.glimit[f] = t->table_rows[f];
    }
    p.sid[f] = storage_of(t, f);
    if (t->pooling && t->pooling[f] == DSF_POOL_MEAN) p.mean_mask |= 1u << f;
  }

  p.F = t->F;
  p.D = t->D;
  p.bf16_tables = t->dtype == DSF_BF16;
}

}  // namespace
}  // namespace bwd
}  // namespace dsf

using namespace dsf;
using namespace dsf::bwd;

extern "C" size_t dsf_bwd_workspace_bytes(int32_t B, int64_t n_values, int64_t n_per_key, int32_t D) {
  if (B < 0 || n_values < 0 || n_values > INT32_MAX || n_per_key < 0 || n_per_key > INT32_MAX ||
      (D != 16 && D != 64))
    return 0;
  return bwd::layout(B, n_values, n_per_key, kMaxF, D).total;
}

extern "C" int dsf_bwd_workspace_offsets(int32_t B, int64_t n_values, int64_t n_per_key, int32_t D,
                                         int64_t* offsets) {
  if (!offsets || dsf_bwd_workspace_bytes(B, n_values, n_per_key, D) == 0) return DSF_EINVAL;
  const bwd::Layout L = bwd::layout(B, n_values, n_per_key, kMaxF, D);
  const size_t at[6] = {L.X, L.H1, L.H2, L.dH2, L.G1, L.dH1};
  for (int i = 0; i < 6; ++i) offsets[i] = static_cast<int64_t>(at[i]);
  return DSF_OK;
}

extern "C" int din_sparse_bwd(const dsf_tables* tables, const dsf_kjt* kjt, const dsf_seq* seq, const int32_t* q_feat,
                              const int32_t* seq_table, int32_t B, const dsf_mlp* mlp, const float* pooled_dev,
                              const float* dpooled_dev, const float* ddin_dev, const dsf_mlp_grads* mg,
                              const dsf_row_grads* rg, void* workspace_dev, size_t ws_bytes, int32_t* status_dev,
                              void* stream) {
  int rc;
  if ((rc = check_tables(tables)) != DSF_OK) return rc;
  if (B < 0 || B > (1 << 24)) return DSF_EINVAL;
  if ((rc = check_kjt(kjt, B, tables->F)) != DSF_OK) return rc;
  if ((rc = check_seq(seq, B)) != DSF_OK) return rc;
  if ((rc = check_mlp(mlp, tables->D)) != DSF_OK) return rc;
  if (!q_feat || !seq_table) return DSF_EINVAL;
  for (int k = 0; k < 3; ++k)
    if (q_feat[k] < 0 || q_feat[k] >= tables->F || seq_table[k] < 0 || seq_table[k] >= tables->F) return DSF_EINVAL;
  if (!pooled_dev || !ddin_dev || !aligned(pooled_dev, 16) || !aligned(ddin_dev, 16)) return DSF_EINVAL;
  if (dpooled_dev && !aligned(dpooled_dev, 16)) return DSF_EINVAL;
  if (!mg || !mg->dW1 || !mg->db1 || !mg->dW2 || !mg->db2 || !mg->dw3 || !mg->db3) return DSF_EINVAL;
  if (!rg || !rg->grad || !rg->touched || !rg->list || !rg->count || rg->list_cap < 0) return DSF_EINVAL;
  if ((rc = check_row_state(tables, rg->grad, rg->touched)) != DSF_OK) return rc;
  const long long Pc = seq->n_per_key;
  const bwd::Layout L = bwd::layout(B, kjt->n_values, Pc, kMaxF, tables->D);
  if (!workspace_dev || !aligned(workspace_dev, 256) || ws_bytes < L.total) return DSF_EWORKSPACE;
  if (B == 0) return DSF_OK;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(workspace_dev);
  const int D = tables->D, F = tables->F, K1 = 12 * D;
  const bool bf = mlp->mode == DSF_MODE_BF16_TC;

  Params p{};
  fill_tables(p, tables);
  p.B = B;
  p.max_len = seq->max_len;
  p.values = reinterpret_cast<const long long*>(kjt->values_dev);
  p.n_values = kjt->n_values;
  p.seq_values = reinterpret_cast<const long long*>(seq->values_dev);
  p.n_seq = seq->n_per_key;
  for (int k = 0; k < 3; ++k) p.q_feat[k] = q_feat[k], p.seq_table[k] = seq_table[k];
  p.bf16_mlp = bf;
  for (int f = 0; f < F; ++f) {
    p.grad[f] = rg->grad[f];
    p.touched[f] = rg->touched[f];
  }
  p.list = reinterpret_cast<long long*>(rg->list);
  p.count = rg->count;
  p.list_cap = rg->list_cap;
  p.status = status_dev;

  long long* boff = reinterpret_cast<long long*>(w + L.boff);
  long long* soff = reinterpret_cast<long long*>(w + L.soff);
  long long* roff = reinterpret_cast<long long*>(w + L.roff);
  int* samp = reinterpret_cast<int*>(w + L.samp);
  float* zb = reinterpret_cast<float*>(w + L.zb);
  float* dab = reinterpret_cast<float*>(w + L.dab);
  float* S = reinterpret_cast<float*>(w + L.S);
  float* G1 = reinterpret_cast<float*>(w + L.G1);
  float* H2 = reinterpret_cast<float*>(w + L.H2);
  float* dX = reinterpret_cast<float*>(w + L.dX);
  float* dS = reinterpret_cast<float*>(w + L.dS);
  void* X = w + L.X;
  void* H1 = w + L.H1;
  void* dH2 = w + L.dH2;
  void* dH1 = w + L.dH1;
  const void* W1 = mlp->W1;
  const void* W2 = mlp->W2;

  float* gbag = reinterpret_cast<float*>(w + L.gbag);
  unsigned long long* okey = reinterpret_cast<unsigned long long*>(w + L.okey);
  long long* osrc = reinterpret_cast<long long*>(w + L.osrc);
  long long* tsum = reinterpret_cast<long long*>(w + L.tsum);
  float* part1 = reinterpret_cast<float*>(w + L.part1);
  float* red = reinterpret_cast<float*>(w + L.red);
  float* part2 = reinterpret_cast<float*>(w + L.part2);
  // the side stream (s2) takes the KJT offsets and the weight packing; the
  // call's stream joins it before the first product
  int dev = 0;
  cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &capturing) != cudaSuccess) return DSF_ECUDA;
  cudaStream_t s2 =
      cudaGetDevice(&dev) == cudaSuccess ? side_stream(dev, capturing == cudaStreamCaptureStatusNone) : nullptr;
  if (!s2 || !follow(s2, s)) s2 = s;
  {  // bag offsets of the KJT (s2); raw and clamped sequence offsets (s)
    const int nk = F * B, tk = (nk + kScanTile - 1) / kScanTile, ts = (B + kScanTile - 1) / kScanTile;
    ScanJobs kj{}, sj{};
    kj.j[0] = ScanJob{kjt->lengths_dev, nk, INT_MAX, tk, tsum, boff, nullptr};
    sj.j[0] = ScanJob{seq->lengths_dev, B, seq->max_len, ts, tsum + 2 * (tk + 1), roff, soff};
    if (tk > 0) {
      scan_tiles_kernel<<<tk, kScanThreads, 0, s2>>>(kj);
      scan_apply_kernel<<<tk, kScanThreads, 0, s2>>>(kj);
      // the occurrence keys of the KJT's values (for the row gradients)
      kjt_keys_kernel<<<grid_for(nk, 256, kMaxBlocks), 256, 0, s2>>>(p, boff, okey, osrc);
    }
    scan_tiles_kernel<<<ts, kScanThreads, 0, s>>>(sj);
    scan_apply_kernel<<<ts, kScanThreads, 0, s>>>(sj);
  }
  // bf16 with x at most 256 wide (D = 16): ds and the dq terms in the dx
  // product's epilogue (dx itself is not written)
  const bool fuse_dsdq = bf && K1 <= 256;
  if (bf) {
    pack_kernel<__nv_bfloat16><<<grid_for(kN1 * K1 + kN2 * kN1, 256), 256, 0, s2>>>(
        mlp->W1, mlp->W2, K1, reinterpret_cast<__nv_bfloat16*>(w + L.w1b), reinterpret_cast<__nv_bfloat16*>(w + L.w2b),
        reinterpret_cast<__nv_bfloat16*>(w + L.w1t), reinterpret_cast<__nv_bfloat16*>(w + L.w2t), fuse_dsdq);
    W1 = w + L.w1b;
    W2 = w + L.w2b;
  } else {
    pack_kernel<float><<<grid_for(kN1 * K1 + kN2 * kN1, 256), 256, 0, s2>>>(
        mlp->W1, mlp->W2, K1, nullptr, nullptr, reinterpret_cast<float*>(w + L.w1t), reinterpret_cast<float*>(w + L.w2t),
        false);
  }
  const void* W1T = w + L.w1t;
  const void* W2T = w + L.w2t;
  if (cudaGetLastError() != cudaSuccess) return DSF_ECUDA;
  // D = A B^T (both row-major with K contiguous), on this library's GEMMs;
  // splits > 1 writes per-split partials to the split buffer
  const int esz = bf ? 2 : 4;
  auto mm = [&](const void* A, long long lda, const void* Bm, long long ldb, float* D, long long ldd, long long M,
                int N, long long K, int splits, const gemm::TnArgs* epi = nullptr) -> bool {
    gemm::TnArgs g = epi ? *epi : gemm::TnArgs{};
    g.A = A;
    g.lda = lda;
    g.B = Bm;
    g.ldb = ldb;
    g.D = D;
    g.ldd = ldd;
    g.M = M;
    g.N = N;
    g.K = K;
    g.k_per_split = ((K + splits - 1) / splits + 63) / 64 * 64;
    if (g.k_per_split < 64) g.k_per_split = 64;
    g.split_stride = M * ldd;
    g.status = status_dev;
    const int n_split = int((K + g.k_per_split - 1) / g.k_per_split);
    return gemm::tn(g, n_split < 1 ? 1 : n_split, bf, s);
  };
  // a sum over all positions: split over K, partials reduced in split order
  const long long P8 = (Pc + 7) / 8 * 8;
  // D [M][N] = A^T B over the K = P positions: bf16 reads the activations as
  // stored, one row per position (A [K][lda], B [K][ldb]); fp32 takes their
  // transposes (A [M][P8], B [N][P8]) on the CUDA cores
  auto mm_splitk = [&](const void* A, long long lda, const void* Bm, long long ldb, float* D, int M, int N,
                       long long K) -> bool {
    // K-splits of at least 256 positions, about kSplitCtas CTAs in all
    const int mt = (M + 127) / 128;
    int splits = int((K + 255) / 256);
    if (splits > kSplitCtas / mt) splits = kSplitCtas / mt;
    if (splits < 1) splits = 1;
    const long long kps = ((K + splits - 1) / splits + 63) / 64 * 64;
    splits = int((K + kps - 1) / kps);
    if (splits < 1) splits = 1;
    float* part = reinterpret_cast<float*>(w + L.split);
    gemm::TnArgs g{};
    g.A = A;
    g.lda = lda;
    g.B = Bm;
    g.ldb = ldb;
    g.D = part;
    g.ldd = N;
    g.M = M;
    g.N = N;
    g.K = K;
    g.k_per_split = kps;
    g.split_stride = (long long)M * N;
    g.status = status_dev;
    const bool ok = bf ? gemm::atb(g, splits, s) : gemm::tn(g, splits, false, s);
    return ok && gemm::reduce(part, (long long)M * N, splits, N, D, N, M, N, s);
  };
  if (Pc > 0) {
    const int gb = grid_for(B, kSampleWarps, kSampleBlocks);
    if (bf)
      gather_kernel<__nv_bfloat16><<<gb, kSampleWarps * 32, 0, s>>>(p, pooled_dev, soff, roff, samp,
                                                                      static_cast<__nv_bfloat16*>(X), S, Pc, okey, osrc);
    else
      gather_kernel<float><<<gb, kSampleWarps * 32, 0, s>>>(p, pooled_dev, soff, roff, samp, static_cast<float*>(X),
                                                              S, Pc, okey, osrc);
    if (cudaGetLastError() != cudaSuccess) return DSF_ECUDA;
  }
  if (!follow(s, s2)) return DSF_ECUDA;  // (the packed weights, the KJT offsets and keys)
  if (Pc > 0) {
    // recompute: h1 = ReLU(x W1^T + b1) (in bf16 mode inside the product's
    // epilogue, which also records h1 > 0 as bits), then the layer-2
    // pre-activation
    if (bf) {
      gemm::TnArgs e{};
      e.epi = gemm::kEpiReluBias;
      e.bias = mlp->b1;
      e.H = H1;
      e.ldh = kN1;
      e.mask = reinterpret_cast<uint32_t*>(w + L.M1);
      e.ldm = kN1 / 32;
      if (!mm(X, K1, W1, K1, nullptr, kN1, Pc, kN1, K1, 1, &e)) return DSF_ECUDA;
    } else {
      if (!mm(X, K1, W1, K1, G1, kN1, Pc, kN1, K1, 1)) return DSF_ECUDA;
      relu1_kernel<float><<<grid_for(Pc * kN1 / 4, 256), 256, 0, s>>>(G1, mlp->b1, static_cast<float*>(H1),
                                                                      Pc * kN1 / 4);
    }
    if (!mm(H1, kN1, W2, kN1, H2, kN2, Pc, kN2, kN1, 1)) return DSF_ECUDA;
  }
  const int smb = grid_for(B, 1, kSampleBlocks);  // (one warp per block)
  if (bf)
    softmax_bwd_kernel<__nv_bfloat16><<<smb, 32, 0, s>>>(p, soff, H2, S, ddin_dev, mlp->b2, mlp->w3, mlp->b3, zb, dab,
                                                         static_cast<__nv_bfloat16*>(dH2), dS, part1, Pc);
  else
    softmax_bwd_kernel<float><<<smb, 32, 0, s>>>(p, soff, H2, S, ddin_dev, mlp->b2, mlp->w3, mlp->b3, zb, dab,
                                                 static_cast<float*>(dH2), dS, part1, Pc);
  if (cudaGetLastError() != cudaSuccess) return DSF_ECUDA;
  if (Pc > 0) {
    // dh1 = (dh2 W2) [h1 > 0] and db1's partial sums (in bf16 mode inside the
    // product's epilogue)
    int rb;
    if (bf) {
      gemm::TnArgs e{};
      e.epi = gemm::kEpiMask;
      e.H = dH1;
      e.ldh = kN1;
      e.mask = reinterpret_cast<uint32_t*>(w + L.M1);
      e.ldm = kN1 / 32;
      e.part = part2;
      if (!mm(dH2, kN2, W2T, kN2, G1, kN1, Pc, kN1, kN2, 1, &e)) return DSF_ECUDA;
      rb = int(4 * ((Pc + 127) / 128));
    } else {
      if (!mm(dH2, kN2, W2T, kN2, G1, kN1, Pc, kN1, kN2, 1)) return DSF_ECUDA;
      rb = grid_for(Pc, 1, kMaxBlocks);
      relu1_bwd_kernel<float><<<rb, kN1, 0, s>>>(G1, static_cast<const float*>(H1), static_cast<float*>(dH1), part2,
                                                 Pc);
    }
    // the bias-gradient columns beside the remaining steps (s2)
    if (!follow(s2, s)) return DSF_ECUDA;
    if (!col_sums(RedJobs{part1, smb, part2, rb, mg->dw3, mg->db2, mg->db3, mg->db1}, red, s2)) return DSF_ECUDA;
    // bf16: the weight gradients (their operands are all written by now) on
    // s2 as well, beside dx, dq/ds and the row gradients
    if (bf) {
      // both products in one launch, kSplitCtas / 3 K-splits each (about
      // kSplitCtas CTAs with equal K-blocks: dW1 has two row tiles, dW2 one),
      // then both reductions in one launch
      int splits = int((Pc + 255) / 256);
      if (splits > kSplitCtas / 3) splits = kSplitCtas / 3;
      if (splits < 1) splits = 1;
      const long long kps = ((Pc + splits - 1) / splits + 63) / 64 * 64;
      splits = int((Pc + kps - 1) / kps);
      if (splits < 1) splits = 1;
      float* part0 = reinterpret_cast<float*>(w + L.split);
      float* part1 = part0 + size_t(splits) * kN1 * K1;
      gemm::TnArgs g0{}, g1{};
      g0.A = dH1, g0.lda = kN1, g0.B = X, g0.ldb = K1, g0.D = part0, g0.ldd = K1, g0.M = kN1, g0.N = K1;
      g1.A = dH2, g1.lda = kN2, g1.B = H1, g1.ldb = kN1, g1.D = part1, g1.ldd = kN1, g1.M = kN2, g1.N = kN1;
      for (gemm::TnArgs* g : {&g0, &g1}) {
        g->K = Pc;
        g->k_per_split = kps;
        g->split_stride = g->M * g->N;
        g->status = status_dev;
      }
      if (!gemm::atb2(g0, splits, g1, splits, s2) ||
          !gemm::reduce2(part0, g0.split_stride, splits, K1, mg->dW1, K1, kN1, K1, part1, g1.split_stride, splits, kN1,
                         mg->dW2, kN1, kN2, kN1, s2))
        return DSF_ECUDA;
    }
    if (fuse_dsdq) {
      gemm::TnArgs e{};
      e.epi = gemm::kEpiDsDq;
      e.nvalid = soff + B;
      e.samp = samp;
      e.S = S;
      e.dS = dS;
      e.dqc = dX;  // (the dq terms, [Pc][Q], in dx's buffer)
      e.pooled = pooled_dev;
      e.pooled_ld = F * D;
      e.dim = D;
      for (int k = 0; k < 3; ++k) e.qoff[k] = q_feat[k] * D;
      if (!mm(dH1, kN1, W1T, kN1, nullptr, K1, Pc, K1, kN1, 1, &e)) return DSF_ECUDA;
    } else {
      if (!mm(dH1, kN1, W1T, kN1, dX, K1, Pc, K1, kN1, 1)) return DSF_ECUDA;
    }
    // the weight gradients (fp32: on transposed copies; bf16: on s2, above)
    if (!bf) {
      void* XT = w + L.XT;
      void* H1T = w + L.H1T;
      void* dH2T = w + L.dH2T;
      void* dH1T = w + L.dH1T;
      if (!gemm::transpose(X, K1, Pc, K1, XT, P8, esz, s) || !gemm::transpose(dH2, kN2, Pc, kN2, dH2T, P8, esz, s) ||
          !gemm::transpose(dH1, kN1, Pc, kN1, dH1T, P8, esz, s) || !gemm::transpose(H1, kN1, Pc, kN1, H1T, P8, esz, s))
        return DSF_ECUDA;
      if (!mm_splitk(dH1T, P8, XT, P8, mg->dW1, kN1, K1, Pc)) return DSF_ECUDA;
      if (!mm_splitk(dH2T, P8, H1T, P8, mg->dW2, kN2, kN1, Pc)) return DSF_ECUDA;
    }
  } else {
    if (cudaMemsetAsync(mg->dW1, 0, size_t(kN1) * K1 * 4, s) != cudaSuccess ||
        cudaMemsetAsync(mg->dW2, 0, size_t(kN2) * kN1 * 4, s) != cudaSuccess ||
        cudaMemsetAsync(mg->db1, 0, size_t(kN1) * 4, s) != cudaSuccess)
      return DSF_ECUDA;
    if (!col_sums(RedJobs{part1, smb, nullptr, 0, mg->dw3, mg->db2, mg->db3, nullptr}, red, s)) return DSF_ECUDA;
  }
  {
    dsdq_kernel<<<grid_for(B, kSampleWarps, kSampleBlocks), kSampleWarps * 32, 0, s>>>(p, boff, soff, roff, Pc, pooled_dev, dpooled_dev, dX, S, dS, gbag,
                                                   fuse_dsdq && Pc > 0 ? dX : nullptr);
    const long long nocc = kjt->n_values + 3 * Pc;
    if (nocc > 0)
      rowgrad_kernel<<<int((nocc + kTile - 1) / kTile), kRowThreads, 0, s>>>(p, boff, soff, Pc, okey, osrc, gbag, dS);
  }
  if (cudaGetLastError() != cudaSuccess || !follow(s, s2)) return DSF_ECUDA;
  return DSF_OK;
}

extern "C" int emb_adagrad_update(const dsf_tables* tables, float* const* accum, const dsf_row_grads* rg, float lr,
                                  float eps, int32_t* status_dev, void* stream) {
  int rc;
  if ((rc = check_tables(tables)) != DSF_OK) return rc;
  if (!accum || !rg || !rg->grad || !rg->touched || !rg->list || !rg->count || rg->list_cap < 0) return DSF_EINVAL;
  if (!(lr >= 0.f) || !(eps >= 0.f)) return DSF_EINVAL;
  if ((rc = check_row_state(tables, rg->grad, rg->touched)) != DSF_OK) return rc;
  if ((rc = check_row_state(tables, accum, nullptr)) != DSF_OK) return rc;
  Params p{};
  fill_tables(p, tables);
  Upd u{};
  for (int f = 0; f < tables->F; ++f) {
    u.table[f] = const_cast<void*>(p.tables[f]);
    u.accum[f] = accum[f];
    u.grad[f] = rg->grad[f];
    u.touched[f] = rg->touched[f];
  }
  u.list = reinterpret_cast<const long long*>(rg->list);
  u.count = rg->count;
  u.cap = rg->list_cap;
  u.D = tables->D;
  u.lr = lr;
  u.eps = eps;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the grid covers the largest possible list; threads past the count exit
  const int g = grid_for(rg->list_cap * (tables->D / 4), 256, 152 * 8);
  if (tables->dtype == DSF_BF16) update_kernel<true><<<g, 256, 0, s>>>(u);
  else update_kernel<false><<<g, 256, 0, s>>>(u);
  reset_count_kernel<<<1, 1, 0, s>>>(rg->count);
  (void)status_dev;
  return cudaGetLastError() == cudaSuccess ? DSF_OK : DSF_ECUDA;
}
