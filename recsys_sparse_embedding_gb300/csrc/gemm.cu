// The backward's matrix products (see gemm.cuh).
#include "gemm.cuh"

#include <cstdint>

#include "dinsparse.h"
#include "ptx.cuh"

namespace dsf {
namespace gemm {
namespace {

constexpr int kThreads = 128;  // 4 warps, one per tensor-memory lane quarter
constexpr int kBM = 128, kBK = 64, kStages = 3;
constexpr int kMaxGridY = 65535;

__device__ __forceinline__ void set_flag(int* status, int bits) {
  if (status && bits) atomicOr(status, bits);
}

template <int BN>
struct Tile {
  static constexpr int A_BYTES = kBM * 128;  // a 128 x 64 bf16 K-block
  static constexpr int B_BYTES = BN * 128;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int EPI_BYTES = 4 * BN * 4;  // the epilogue's per-warp column sums
  static constexpr int BODY = kStages * STAGE > EPI_BYTES ? kStages * STAGE : EPI_BYTES;
  static constexpr int SMEM = BODY + 1024;  // + alignment slack
  static constexpr uint32_t TCOLS = BN <= 64 ? 64 : (BN <= 128 ? 128 : 256);
  static_assert(BN % 16 == 0 && BN >= 32 && BN <= 256, "tcgen05 N for M = 128");
  static_assert(STAGE % 1024 == 0, "stages keep the 1024-byte swizzle-atom alignment");
};

__device__ __forceinline__ uint32_t bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// The epilogue of one 128-row tile whose accumulator (BN columns) starts at
// tensor-memory column tbase. Thread t owns row t of the tile (its lane of
// tensor memory) and walks its row 16 columns at a time, straight from
// registers: the fp32 row of D (nullable), the fused transform of a.epi, the
// bf16 row of H, and its transposed copy HT (2-byte stores: the 32 lanes of a
// warp hold 32 consecutive rows, so each store instruction writes 64
// contiguous bytes of one HT row). kEpiMask's column sums go through a
// fixed-order shuffle tree per warp and a four-warp sum in shared memory
// (csum: 4 * BN floats). have_acc false: the product is zero.
template <int BN>
__device__ __forceinline__ void epilogue(const TnArgs& a, float* csum, uint32_t tbase, long long m0, long long tile,
                                         float* D, bool have_acc) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long row = m0 + tid;
  const bool live = row < a.M;
  __nv_bfloat16* H = static_cast<__nv_bfloat16*>(a.H);
  __nv_bfloat16* HT = static_cast<__nv_bfloat16*>(a.HT);
  const __nv_bfloat16* Hin = static_cast<const __nv_bfloat16*>(a.Hin);
  const int nlim = a.N < BN ? a.N : BN;
#pragma unroll 1
  for (int c0 = 0; c0 < nlim; c0 += 16) {
    float v[16];
    uint4 hin0 = make_uint4(0u, 0u, 0u, 0u), hin1 = hin0;
    if (a.epi == kEpiMask && live) {  // (issued before the tensor-memory load)
      hin0 = *reinterpret_cast<const uint4*>(Hin + row * a.ldh + c0);
      hin1 = *reinterpret_cast<const uint4*>(Hin + row * a.ldh + c0 + 8);
    }
    if (have_acc) {
      tmem_ld16(tbase + (uint32_t(warp * 32) << 16) + uint32_t(c0), v);
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = 0.f;
    }
    const bool full = c0 + 16 <= a.N;
    if (D && live) {
      float* d = D + row * a.ldd + c0;
      if (full && (reinterpret_cast<uintptr_t>(d) & 15) == 0) {
#pragma unroll
        for (int j = 0; j < 16; j += 4) *reinterpret_cast<float4*>(d + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
      } else {
        for (int j = 0; j < 16 && c0 + j < a.N; ++j) d[j] = v[j];
      }
    }
    if (a.epi == kEpiF32) continue;
    if (a.epi == kEpiReluBias) {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = fmaxf(v[j] + __ldg(a.bias + c0 + j), 0.f);
    } else {
      const uint32_t hw[8] = {hin0.x, hin0.y, hin0.z, hin0.w, hin1.x, hin1.y, hin1.z, hin1.w};
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        if (!(bf16_lo(hw[t]) > 0.f)) v[2 * t] = 0.f;
        if (!(bf16_hi(hw[t]) > 0.f)) v[2 * t + 1] = 0.f;
      }
    }
    uint32_t packed[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) packed[t] = bf16x2(v[2 * t], v[2 * t + 1]);
    if (live) {
      *reinterpret_cast<uint4*>(H + row * a.ldh + c0) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      *reinterpret_cast<uint4*>(H + row * a.ldh + c0 + 8) = make_uint4(packed[4], packed[5], packed[6], packed[7]);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint16_t b16 = uint16_t(j & 1 ? packed[j >> 1] >> 16 : packed[j >> 1] & 0xffffu);
        reinterpret_cast<uint16_t*>(HT)[(long long)(c0 + j) * a.ldt + row] = b16;
      }
    }
    if (a.epi == kEpiMask && a.part) {
      // the warp's column sums of the masked values (rows past M are zero),
      // a fixed-order tree over the lanes
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float x = v[j];
#pragma unroll
        for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) csum[warp * BN + c0 + j] = x;
      }
    }
  }
  if (a.epi == kEpiMask && a.part) {
    __syncthreads();
    for (int c = tid; c < nlim; c += kThreads)
      a.part[tile * a.N + c] = ((csum[c] + csum[BN + c]) + csum[2 * BN + c]) + csum[3 * BN + c];
    __syncthreads();
  }
}

// D (+ split) = A[m0 : m0 + 128][k-range] * B[0 : BN][k-range]^T, bf16, with
// the epilogue a.epi.
template <int BN>
__global__ void __launch_bounds__(kThreads, 1) tn_bf16_kernel(const TnArgs a) {
  using T = Tile<BN>;
  extern __shared__ uint8_t dyn[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar[kStages];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long m0 = (long long)blockIdx.x * kBM;
  const long long k0 = (long long)blockIdx.y * a.k_per_split;
  const long long k1 = k0 + a.k_per_split < a.K ? k0 + a.k_per_split : a.K;
  const int nkb = k1 > k0 ? int((k1 - k0 + kBK - 1) / kBK) : 0;
  float* D = a.D ? a.D + (long long)blockIdx.y * a.split_stride : nullptr;
  const __nv_bfloat16* A = static_cast<const __nv_bfloat16*>(a.A);
  const __nv_bfloat16* Bm = static_cast<const __nv_bfloat16*>(a.B);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
    fence_mbarrier_init();
    abort_ = 0;
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, T::TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;

  // K-block kb into its stage: 16-byte chunks in the 128-byte swizzle layout
  // (chunk c of row r at r * 128 + (c ^ (r % 8)) * 16); rows past M or N and
  // elements past the split's K-range are zero-filled.
  auto load = [&](int kb) {
    uint8_t* sa = sm + (kb % kStages) * T::STAGE;
    uint8_t* sb = sa + T::A_BYTES;
    const long long kk = k0 + (long long)kb * kBK;
    for (int q = tid; q < kBM * 8; q += kThreads) {
      const int r = q >> 3, c = q & 7;
      const long long row = m0 + r, k = kk + c * 8;
      long long v = row < a.M ? k1 - k : 0;
      v = v < 0 ? 0 : (v > 8 ? 8 : v);
      const __nv_bfloat16* src = v > 0 ? A + row * a.lda + k : A;
      cp_async_16_ca(sa + r * 128 + ((c ^ (r & 7)) << 4), src, uint32_t(v * 2));
    }
    for (int q = tid; q < BN * 8; q += kThreads) {
      const int r = q >> 3, c = q & 7;
      const long long k = kk + c * 8;
      long long v = r < a.N ? k1 - k : 0;
      v = v < 0 ? 0 : (v > 8 ? 8 : v);
      const __nv_bfloat16* src = v > 0 ? Bm + (long long)r * a.ldb + k : Bm;
      cp_async_16_ca(sb + r * 128 + ((c ^ (r & 7)) << 4), src, uint32_t(v * 2));
    }
  };
  constexpr uint32_t IDESC = idesc_bf16_f32(kBM, BN);
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < nkb) load(s);
    cp_async_commit();
  }
  int issued = -1;  // last K-block whose MMAs were committed
  for (int kb = 0; kb < nkb; ++kb) {
    cp_async_wait_one_pending();  // (kStages - 2 = 1 group may stay in flight)
    fence_proxy_async_smem();
    __syncthreads();
    if (abort_) break;
    if (tid == 0) {
      tc_fence_after();
      const uint32_t sa = smem_u32(sm + (kb % kStages) * T::STAGE), sb = sa + T::A_BYTES;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
        tc_mma_f16(tbase, sw128_kmajor_desc(sa + kk * 32), sw128_kmajor_desc(sb + kk * 32), IDESC,
                   (kb > 0 || kk > 0) ? 1u : 0u);
      tc_commit(&bar[kb % kStages]);
    }
    issued = kb;
    // block kb + kStages - 1 goes into the stage block kb - 1 used: wait for
    // that block's MMAs first (block kb's run meanwhile)
    const int nx = kb + kStages - 1;
    if (nx < nkb) {
      if (kb >= 1) {
        if (tid == 0 && !mbar_wait(&bar[(kb - 1) % kStages], uint32_t(((kb - 1) / kStages) & 1))) abort_ = 1;
        __syncthreads();
      }
      if (!abort_) load(nx);
    }
    cp_async_commit();
  }
  cp_async_wait_all();
  // every MMA done (a commit tracks all earlier MMAs of its thread)
  if (tid == 0 && issued >= 0 && !mbar_wait(&bar[issued % kStages], uint32_t((issued / kStages) & 1))) abort_ = 1;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (!abort_) epilogue<BN>(a, reinterpret_cast<float*>(sm), tbase, m0, blockIdx.x, D, nkb > 0);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, T::TCOLS);
  if (tid == 0 && abort_) set_flag(a.status, DSF_FLAG_TIMEOUT);
}

// B resident: D = A B^T with N <= 256 and K <= 64 * KB <= 256 (B, the MLP
// weights, fits shared memory whole). Persistent CTAs, one per SM, walk the
// 128-row tiles of A; B is loaded once. Per tile: the tile's A has landed ->
// its MMAs -> the next tile's A starts loading -> this tile's epilogue
// (overlapping that load).
template <int BN, int KB>
struct RTile {
  static constexpr int B_BYTES = KB * BN * 128;
  static constexpr int A_BYTES = KB * kBM * 128;
  static constexpr int E_BYTES = 4 * BN * 4;
  static constexpr int SMEM = B_BYTES + A_BYTES + E_BYTES + 1024;
  static constexpr uint32_t TCOLS = BN <= 64 ? 64 : (BN <= 128 ? 128 : 256);
  static_assert(B_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "1024-byte swizzle-atom alignment");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

template <int BN, int KB>
__global__ void __launch_bounds__(kThreads, 1) tn_bf16_resident_kernel(const TnArgs a) {
  using T = RTile<BN, KB>;
  extern __shared__ uint8_t dyn[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = sm;
  uint8_t* sA = sm + T::B_BYTES;
  uint8_t* sE = sA + T::A_BYTES;
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_;
  const int tid = threadIdx.x, warp = tid >> 5;
  const long long tiles = (a.M + kBM - 1) / kBM;
  if ((long long)blockIdx.x >= tiles) return;
  const __nv_bfloat16* A = static_cast<const __nv_bfloat16*>(a.A);
  const __nv_bfloat16* Bm = static_cast<const __nv_bfloat16*>(a.B);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
    abort_ = 0;
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, T::TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_slot;
  // 16-byte chunks in the 128-byte swizzle layout, K-block by K-block;
  // rows past M / N and elements past K are zero-filled
  for (int q = tid; q < KB * BN * 8; q += kThreads) {
    const int kb = q / (BN * 8), rem = q - kb * (BN * 8), r = rem >> 3, c = rem & 7;
    const long long k = (long long)kb * kBK + c * 8;
    long long v = r < a.N ? a.K - k : 0;
    v = v < 0 ? 0 : (v > 8 ? 8 : v);
    const __nv_bfloat16* src = v > 0 ? Bm + (long long)r * a.ldb + k : Bm;
    cp_async_16_ca(sB + kb * (BN * 128) + r * 128 + ((c ^ (r & 7)) << 4), src, uint32_t(v * 2));
  }
  auto load_a = [&](long long t) {
    for (int q = tid; q < KB * kBM * 8; q += kThreads) {
      const int kb = q / (kBM * 8), rem = q - kb * (kBM * 8), r = rem >> 3, c = rem & 7;
      const long long row = t * kBM + r, k = (long long)kb * kBK + c * 8;
      long long v = row < a.M ? a.K - k : 0;
      v = v < 0 ? 0 : (v > 8 ? 8 : v);
      const __nv_bfloat16* src = v > 0 ? A + row * a.lda + k : A;
      cp_async_16_ca(sA + kb * (kBM * 128) + r * 128 + ((c ^ (r & 7)) << 4), src, uint32_t(v * 2));
    }
  };
  load_a(blockIdx.x);
  cp_async_commit();
  constexpr uint32_t IDESC = idesc_bf16_f32(kBM, BN);
  uint32_t phase = 0;
  for (long long t = blockIdx.x; t < tiles; t += gridDim.x) {
    cp_async_wait_all();
    fence_proxy_async_smem();
    __syncthreads();
    if (abort_) break;
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kb = 0; kb < KB; ++kb)
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          tc_mma_f16(tbase, sw128_kmajor_desc(smem_u32(sA + kb * (kBM * 128)) + kk * 32),
                     sw128_kmajor_desc(smem_u32(sB + kb * (BN * 128)) + kk * 32), IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
      tc_commit(&bar);
      if (!mbar_wait(&bar, phase)) abort_ = 1;
    }
    phase ^= 1u;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (abort_) break;
    // the next tile's A streams in while this tile's epilogue runs
    if (t + gridDim.x < tiles) load_a(t + gridDim.x);
    cp_async_commit();
    epilogue<BN>(a, reinterpret_cast<float*>(sE), tbase, t * kBM, t, a.D, true);
    tc_fence_before();  // (this tile's tensor-memory reads before the next tile's MMAs)
  }
  cp_async_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, T::TCOLS);
  if (tid == 0 && abort_) set_flag(a.status, DSF_FLAG_TIMEOUT);
}

// fp32 operands on the CUDA cores: 64 x 64 tiles of D, 256 threads, 4 x 4
// results each; K-steps of 16 staged in shared memory.
__global__ void __launch_bounds__(256) tn_f32_kernel(const TnArgs a, int n0) {
  constexpr int BM = 64, BN = 64, BK = 16;
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const long long m0 = (long long)blockIdx.x * BM;
  const int nb = n0 + blockIdx.z * BN;
  const long long k0 = (long long)blockIdx.y * a.k_per_split;
  const long long k1 = k0 + a.k_per_split < a.K ? k0 + a.k_per_split : a.K;
  const float* A = static_cast<const float*>(a.A);
  const float* Bm = static_cast<const float*>(a.B);
  float* D = a.D + (long long)blockIdx.y * a.split_stride;
  float acc[4][4] = {};
  for (long long kk = k0; kk < k1; kk += BK) {
    // 64 rows x 16 k of A and of B: four elements per thread each
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = tid + i * 256, r = e >> 4, c = e & 15;
      const long long k = kk + c;
      const long long ra = m0 + r;
      const int rb = nb + r;
      As[c][r] = (ra < a.M && k < k1) ? A[ra * a.lda + k] : 0.f;
      Bs[c][r] = (rb < a.N && k < k1) ? Bm[(long long)rb * a.ldb + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < BK; ++c) {
      float x[4], y[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[i] = As[c][ty * 4 + i];
        y[i] = Bs[c][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(x[i], y[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long long row = m0 + ty * 4 + i;
    if (row >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = nb + tx * 4 + j;
      if (col < a.N) D[row * a.ldd + col] = acc[i][j];
    }
  }
}

// 32 consecutive outputs per block of 256 threads: warp g adds splits g,
// g + 8, g + 16, ... in increasing order (eight loads in flight), then warp
// 0 adds the eight warps' sums in warp order. The order is fixed, so the
// result is deterministic.
__global__ void __launch_bounds__(256) reduce_kernel(const float* P, long long split_stride, int splits, long long ldp,
                                                     float* D, long long ldd, long long M, int N) {
  __shared__ float part[8][33];
  const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
  const long long total = M * N;
  for (long long base = blockIdx.x * 32LL; base < total; base += gridDim.x * 32LL) {
    const long long i = base + lane;
    const long long m = i < total ? i / N : 0;
    const int n = int(i - m * N);
    float s = 0.f;
    if (i < total) {
      const float* q = P + m * ldp + n;
      for (int z0 = g; z0 < splits; z0 += 64) {
        float v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) v[t] = z0 + 8 * t < splits ? q[(long long)(z0 + 8 * t) * split_stride] : 0.f;
#pragma unroll
        for (int t = 0; t < 8; ++t)
          if (z0 + 8 * t < splits) s += v[t];
      }
    }
    part[g][lane] = s;
    __syncthreads();
    if (g == 0 && i < total) {
      float r = part[0][lane];
#pragma unroll
      for (int k = 1; k < 8; ++k) r += part[k][lane];
      D[m * ldd + n] = r;
    }
    __syncthreads();
  }
}

// 2-byte elements, 64 x 64 tiles: 16-byte loads (8 consecutive columns of a
// row) and 16-byte stores (8 consecutive rows of a column); both strides
// multiples of 8 elements.
__global__ void transpose16_kernel(const uint16_t* in, long long ld_in, long long rows, int cols, uint16_t* out,
                                   long long ld_out) {
  __shared__ uint16_t t[64][64 + 2];
  const long long r0 = (long long)blockIdx.x * 64;
  const int c0 = blockIdx.y * 64;
  for (int q = threadIdx.x; q < 64 * 8; q += blockDim.x) {
    const int i = q >> 3, j = (q & 7) * 8;
    const long long r = r0 + i;
    uint16_t v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (r < rows) {
      if (c0 + j + 8 <= cols) {
        const uint4 x = *reinterpret_cast<const uint4*>(in + r * ld_in + c0 + j);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) { v[2 * k] = uint16_t(w[k]); v[2 * k + 1] = uint16_t(w[k] >> 16); }
      } else {
        for (int k = 0; c0 + j + k < cols && k < 8; ++k) v[k] = in[r * ld_in + c0 + j + k];
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) t[i][j + k] = v[k];
  }
  __syncthreads();
  for (int q = threadIdx.x; q < 64 * 8; q += blockDim.x) {
    const int j = q >> 3, i = (q & 7) * 8;
    const int c = c0 + j;
    const long long r = r0 + i;
    if (c >= cols || r >= rows) continue;
    if (r + 8 <= rows) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) w[k] = uint32_t(t[i + 2 * k][j]) | (uint32_t(t[i + 2 * k + 1][j]) << 16);
      *reinterpret_cast<uint4*>(out + (long long)c * ld_out + r) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      for (int k = 0; r + k < rows; ++k) out[(long long)c * ld_out + r + k] = t[i + k][j];
    }
  }
}

template <typename E>
__global__ void transpose_kernel(const E* in, long long ld_in, long long rows, int cols, E* out, long long ld_out) {
  __shared__ E t[32][33];
  const long long r0 = (long long)blockIdx.x * 32;
  const int c0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const long long r = r0 + i;
    const int c = c0 + threadIdx.x;
    if (r < rows && c < cols) t[i][threadIdx.x] = in[r * ld_in + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c = c0 + i;
    const long long r = r0 + threadIdx.x;
    if (r < rows && c < cols) out[(long long)c * ld_out + r] = t[threadIdx.x][i];
  }
}

template <int BN>
bool launch_bf16(const TnArgs& a, int splits, cudaStream_t s) {
  using T = Tile<BN>;
  static bool attr_set[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(tn_bf16_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM) !=
        cudaSuccess)
      return false;
    attr_set[dev] = true;
  }
  const long long mt = (a.M + kBM - 1) / kBM;
  if (mt <= 0 || mt > 0x7fffffff || splits < 1 || splits > kMaxGridY) return false;
  tn_bf16_kernel<BN><<<dim3(unsigned(mt), unsigned(splits)), kThreads, T::SMEM, s>>>(a);
  return cudaGetLastError() == cudaSuccess;
}

template <int BN, int KB>
int launch_resident(const TnArgs& a, cudaStream_t s) {  // 1 ok, 0 failed
  using T = RTile<BN, KB>;
  static bool attr_set[64] = {};
  static int nsm[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(tn_bf16_resident_kernel<BN, KB>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&nsm[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    attr_set[dev] = true;
  }
  const long long tiles = (a.M + kBM - 1) / kBM;
  const long long g = tiles < nsm[dev] ? tiles : nsm[dev];
  if (g <= 0) return 1;
  tn_bf16_resident_kernel<BN, KB><<<unsigned(g), kThreads, T::SMEM, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? 1 : 0;
}

}  // namespace

size_t tn_bf16_smem_bytes(int N) {
  if (N <= 64) return Tile<64>::SMEM;
  if (N <= 128) return Tile<128>::SMEM;
  if (N <= 192) return Tile<192>::SMEM;
  return Tile<256>::SMEM;
}

bool tn(const TnArgs& a0, int splits, bool bf16, cudaStream_t s) {
  if (a0.M <= 0 || a0.N <= 0 || a0.K < 0 || splits < 1) return a0.M <= 0 || a0.N <= 0;
  if (a0.k_per_split <= 0 || a0.k_per_split % kBK != 0) return false;
  // (cp.async of 16-byte chunks: bf16 rows must start 16-byte aligned)
  if (bf16 && ((reinterpret_cast<uintptr_t>(a0.A) & 15) || (reinterpret_cast<uintptr_t>(a0.B) & 15) ||
               (a0.lda * 2) % 16 || (a0.ldb * 2) % 16))
    return false;
  if (!bf16) {
    const long long mt = (a0.M + 63) / 64;
    const int nt = (a0.N + 63) / 64;
    if (mt > 0x7fffffff || splits > kMaxGridY || nt > kMaxGridY) return false;
    tn_f32_kernel<<<dim3(unsigned(mt), unsigned(splits), unsigned(nt)), 256, 0, s>>>(a0, 0);
    return cudaGetLastError() == cudaSuccess;
  }
  if (a0.epi != kEpiF32 && (a0.N > 256 || a0.N % 32 != 0 || !a0.H || !a0.HT || a0.ldh % 8 || a0.ldt % 8))
    return false;
  // B resident (the products with a weight matrix as B): persistent CTAs
  if (splits == 1 && a0.K <= 4 * kBK && a0.N <= 256) {
    const int kb = int((a0.K + kBK - 1) / kBK);
    const int bn = a0.N <= 64 ? 64 : (a0.N <= 128 ? 128 : (a0.N <= 192 ? 192 : 256));
    int r = -1;
    if (bn == 64 && kb == 4) r = launch_resident<64, 4>(a0, s);
    else if (bn == 256 && kb == 3) r = launch_resident<256, 3>(a0, s);
    else if (bn == 256 && kb == 1) r = launch_resident<256, 1>(a0, s);
    else if (bn == 192 && kb == 4) r = launch_resident<192, 4>(a0, s);
    else if (bn == 256 && kb == 4) r = launch_resident<256, 4>(a0, s);
    if (r >= 0) return r == 1;
  }
  // N in chunks of at most 256 columns: B's rows and D's columns move on
  for (int n0 = 0; n0 < a0.N; n0 += 256) {
    TnArgs a = a0;
    a.N = a0.N - n0 < 256 ? a0.N - n0 : 256;
    a.B = static_cast<const __nv_bfloat16*>(a0.B) + (long long)n0 * a0.ldb;
    a.D = a0.D + n0;
    bool ok;
    if (a.N <= 64) ok = launch_bf16<64>(a, splits, s);
    else if (a.N <= 128) ok = launch_bf16<128>(a, splits, s);
    else if (a.N <= 192) ok = launch_bf16<192>(a, splits, s);
    else ok = launch_bf16<256>(a, splits, s);
    if (!ok) return false;
  }
  return true;
}

bool reduce(const float* P, long long split_stride, int splits, long long ldp, float* D, long long ldd, long long M,
            int N, cudaStream_t s) {
  const long long total = M * N;
  if (total <= 0) return true;
  long long g = (total + 31) / 32;
  if (g > 152 * 8) g = 152 * 8;
  reduce_kernel<<<unsigned(g), 256, 0, s>>>(P, split_stride, splits, ldp, D, ldd, M, N);
  return cudaGetLastError() == cudaSuccess;
}

bool transpose(const void* in, long long ld_in, long long rows, int cols, void* out, long long ld_out, int esize,
               cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return true;
  const long long gx = (rows + 31) / 32;
  const int gy = (cols + 31) / 32;
  if (gx > 0x7fffffff || gy > kMaxGridY) return false;
  const dim3 grid{static_cast<unsigned>(gx), static_cast<unsigned>(gy), 1u};
  const dim3 block{32u, 8u, 1u};
  if (esize == 2 && ld_in % 8 == 0 && ld_out % 8 == 0 && (reinterpret_cast<uintptr_t>(in) & 15) == 0 &&
      (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
    const long long hx = (rows + 63) / 64;
    const int hy = (cols + 63) / 64;
    if (hx > 0x7fffffff || hy > kMaxGridY) return false;
    transpose16_kernel<<<dim3{static_cast<unsigned>(hx), static_cast<unsigned>(hy), 1u}, 256, 0, s>>>(
        static_cast<const uint16_t*>(in), ld_in, rows, cols, static_cast<uint16_t*>(out), ld_out);
  } else if (esize == 2)
    transpose_kernel<uint16_t><<<grid, block, 0, s>>>(static_cast<const uint16_t*>(in), ld_in, rows, cols,
                                                       static_cast<uint16_t*>(out), ld_out);
  else if (esize == 4)
    transpose_kernel<uint32_t><<<grid, block, 0, s>>>(static_cast<const uint32_t*>(in), ld_in, rows, cols,
                                                       static_cast<uint32_t*>(out), ld_out);
  else
    return false;
  return cudaGetLastError() == cudaSuccess;
}

}  // namespace gemm
}  // namespace dsf
